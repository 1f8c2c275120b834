// prefill_tc_kernel.cuh -- several query rows per sequence on the 5th-generation tensor
// cores (tcgen05), for groups long enough to fill 128-row tiles (chunked prefill).
//
// One CTA (4 warps) per 128 (token, query head) rows of one (sequence, kv head) group,
// the rows packed token-major as in the multi-row decode kernel (AstrAI "CUDA Kernels",
// "Q Scheduling and KV Addressing": the query heads of one kv-head group share each
// K/V tile).  The CTA walks the keys its rows may see in tiles of 128:
//     S  = Q K^T       tcgen05.mma M=128 rows, N=128 keys, K=D; S in tensor memory
//     softmax          thread r owns row r = TMEM lane r: the row max and sums need no
//                      shuffles; the base-2 online recurrence of the decode kernel
//     O += P V         tcgen05.mma M=128 rows, N=D, K=128 keys; O in tensor memory,
//                      rescaled in place (tcgen05.ld/st) only when a warp's running
//                      maximum moved
// Q, K and V tiles sit in shared memory 128B-swizzled, K-major ([D/64][rows][64]) as the
// TMA boxes land them; P is written by the softmax threads in the same layout; V is
// read MN-major (N = dims contiguous).  K/V tiles are double-buffered; one thread
// issues the copies and the MMAs, whose completions arrive on mbarriers
// (tcgen05.commit).  Keys past the sequence's length, or in a page whose id is out of
// range, are masked in the scores and zeroed in V's shared-memory rows (0 * NaN would
// reach the output).  Every wait is bounded; on a timeout the status word is set, the
// CTA stops issuing work and releases its tensor memory.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pkv.h"
#include "ptx.cuh"

namespace pkv {

struct PrefillTcParams {
    const __nv_bfloat16 *q;  // [total_q, Hq, D]
    const int *qo_indptr;    // [B+1]
    const int *block_table;  // [B, max_pages]
    const int *seq_lens;     // [B]
    __nv_bfloat16 *out;      // [total_q, Hq, D]
    float *lse;              // [total_q, Hq] or nullptr
    int *status;
    int B, Hq, Hkv, G, P, log2P, num_pages, max_pages, total_q, max_q_len, causal, q_tiles;
    float scale_log2;
    unsigned long long wait_limit_ns;
};

constexpr int kTcRows = 128;  // rows per CTA (the MMA's M)
constexpr int kTcKeys = 128;  // keys per tile (the score MMA's N)

// Shared memory (bytes from a 1024-aligned base) of the D = 128 kernel.
struct TcSmem {
    static constexpr int kTile = kTcRows * 128 * 2;  // 128 rows x 128 dims bf16, as 2 column blocks
    static constexpr int q = 0, p = kTile;
    static constexpr int kv = 2 * kTile;             // stage s: K at kv + s*2*kTile, V 1 tile after
    static constexpr int bars = 6 * kTile;           // 2 copy barriers, S done, O done
    static constexpr int ok = bars + 64;             // [2 stages][16 boxes] page-valid flags
    static constexpr int tmem_slot = ok + 2 * 16 * 4;
    static constexpr int total = tmem_slot + 16;
    static constexpr int dynamic = total + 1024;
};

__global__ void __launch_bounds__(128, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const PrefillTcParams p)
{
    constexpr int D = 128;
    constexpr int kTile = TcSmem::kTile;
    constexpr int kBlk = kTcRows * 128;  // bytes of one 64-column block of a tile
    const int kvh = (int)(blockIdx.x % (unsigned)p.Hkv), qt = (int)(blockIdx.x / (unsigned)p.Hkv);
    const int b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G;

    if (tid == 0) {
        prefetch_tensor_map(&tmK);
        prefetch_tensor_map(&tmV);
    }
    griddep_wait();

    const int q_base = p.qo_indptr[b];
    const int n_q = p.qo_indptr[b + 1] - q_base;
    if (q_base < 0 || n_q < 0 || n_q > p.max_q_len || q_base + n_q > p.total_q) {
        if (tid == 0 && kvh == 0 && qt == 0) atomicCAS(p.status, 0, PKV_ERR_BAD_QO_INDPTR);
        return;
    }
    const int row0 = qt * kTcRows;
    const int nrows = min(kTcRows, n_q * G - row0);
    if (nrows <= 0) return;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_pages * p.P) {
        if (tid == 0 && kvh == 0 && qt == 0) atomicCAS(p.status, 0, PKV_ERR_BAD_SEQ_LEN);
        L = 0;
    }
    // this thread's row: token, head, global row, last key it may see
    const int r = tid;
    const bool row_ok = r < nrows;
    const int tok = (row0 + (row_ok ? r : 0)) / G, head = (row0 + (row_ok ? r : 0)) % G;
    const size_t grow = (size_t)(q_base + tok) * p.Hq + kvh * G + head;
    const int klim = p.causal ? L - n_q + tok : L - 1;
    // keys any row of the CTA may see
    const int last_tok = (row0 + nrows - 1) / G;
    const int n_keys = max(0, p.causal ? min(L, L - n_q + last_tok + 1) : L);
    const int n_tiles = (n_keys + kTcKeys - 1) / kTcKeys;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *sbase = smem_raw + (base - raw_addr);
    const uint32_t sQ = base + TcSmem::q, sP = base + TcSmem::p;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + TcSmem::bars);
    int *sm_ok = reinterpret_cast<int *>(sbase + TcSmem::ok);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + TcSmem::tmem_slot);
    const uint32_t bar_full0 = smem_addr(&bars[0]), bar_s = smem_addr(&bars[2]), bar_o = smem_addr(&bars[3]);
    auto sK = [&](int st) { return base + TcSmem::kv + (uint32_t)(st * 2 * kTile); };
    auto sV = [&](int st) { return sK(st) + (uint32_t)kTile; };

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_barrier_init();
    }
    if (warp == 0) tc_alloc(smem_addr(tmem_slot), 256);  // S: columns 0..127, O: 128..255

    // Q rows into shared memory, 128B-swizzled [2 column blocks][128 rows][128 B]
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.q + grow * D);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint4 v = row_ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            const int dc = c >> 3, cc = c & 7;
            st_shared_v4(sQ + (uint32_t)(dc * kBlk + r * 128 + ((cc ^ (r & 7)) << 4)), v.x, v.y, v.z, v.w);
        }
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128u;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    const uint64_t policy = l2_policy_evict_first();
    const int box_t = p.P < kTcKeys ? p.P : kTcKeys;
    const int nbox = kTcKeys / box_t;
    // copies of key tile j into stage st (thread 0)
    auto issue = [&](int j, int st) {
        const uint32_t bar = bar_full0 + 8u * (uint32_t)st;
        uint32_t bytes = 0;
        int ids[16];
        for (int x = 0; x < nbox; ++x) {
            const int key = j * kTcKeys + x * box_t;
            int pg = -1;
            if (key < n_keys) {
                pg = p.block_table[(size_t)b * p.max_pages + (key >> p.log2P)];
                if ((unsigned)pg >= (unsigned)p.num_pages) {
                    atomicCAS(p.status, 0, PKV_ERR_BAD_PAGE_INDEX);
                    pg = -1;
                }
            }
            ids[x] = pg;
            sm_ok[st * 16 + x] = pg >= 0;
            if (pg >= 0) bytes += 2u * 2u * (uint32_t)box_t * 128u;
        }
        mbar_arrive_expect_tx(bar, bytes);
        for (int x = 0; x < nbox; ++x) {
            if (ids[x] < 0) continue;
            const int key = j * kTcKeys + x * box_t;
            const int row = ids[x] * p.P + (key & (p.P - 1));
#pragma unroll
            for (int dc = 0; dc < 2; ++dc) {
                const uint32_t off = (uint32_t)(dc * kBlk + x * box_t * 128);
                tma_load_3d(sK(st) + off, &tmK, dc * 64, kvh, row, bar, policy);
                tma_load_3d(sV(st) + off, &tmV, dc * 64, kvh, row, bar, policy);
            }
        }
    };
    if (tid == 0) {
        if (n_tiles > 0) issue(0, 0);
        if (n_tiles > 1) issue(1, 1);
    }

    float m_run = -__int_as_float(0x7f800000), l_run = 0.f, lt_run = 0.f;
    bool failed = false;
    constexpr uint32_t kIdS = tc_idesc_bf16(kTcRows, kTcKeys, false);
    constexpr uint32_t kIdO = tc_idesc_bf16(kTcRows, D, true);
    for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        const bool got = mbar_wait_bounded(bar_full0 + 8u * (uint32_t)st, ph, p.wait_limit_ns);
        if (!__syncthreads_and(got)) {
            failed = true;
            break;
        }
        // keys of this tile that are not valid: zero their V rows (0 * NaN would reach O)
        const bool tail = (j + 1) * kTcKeys > n_keys;
        int bad_box = 0;
        for (int x = 0; x < nbox; ++x) bad_box |= !sm_ok[st * 16 + x];
        if (tail || bad_box) {
            const int key = j * kTcKeys + r;
            if (key >= n_keys || !sm_ok[st * 16 + r / box_t]) {
#pragma unroll
                for (int dc = 0; dc < 2; ++dc)
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        st_shared_v4(sV(st) + (uint32_t)(dc * kBlk + r * 128 + cc * 16), 0u, 0u, 0u, 0u);
            }
            fence_proxy_async_shared();
            __syncthreads();
        }
        // S = Q K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int dc = 0; dc < 2; ++dc)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc_mma_bf16(tS, tc_desc(sQ + (uint32_t)(dc * kBlk + k * 32), 16, 1024),
                                tc_desc(sK(st) + (uint32_t)(dc * kBlk + k * 32), 16, 1024), kIdS, (dc | k) != 0);
            tc_commit(bar_s);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar_s, (uint32_t)(j & 1), p.wait_limit_ns))) {
            failed = true;
            break;
        }
        tc_fence_after();
        // softmax of this thread's row over the tile's 128 keys
        float sv[kTcKeys];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            tc_ld32(tS + lane_off + (uint32_t)(cb * 32), v);
#pragma unroll
            for (int i = 0; i < 32; ++i) sv[cb * 32 + i] = v[i];
        }
        const int key0 = j * kTcKeys;
        const int lim = row_ok ? klim : -1;  // the last key this row sees (rows past the group see none)
        float mx = -__int_as_float(0x7f800000);
        if (tail || bad_box) {
#pragma unroll
            for (int i = 0; i < kTcKeys; ++i) {
                const int key = key0 + i;
                float v = sv[i] * p.scale_log2;
                if (key > lim || key >= n_keys || !sm_ok[st * 16 + i / box_t]) v = -__int_as_float(0x7f800000);
                sv[i] = v;
                mx = fmaxf(mx, v);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kTcKeys; ++i) {
                float v = sv[i] * p.scale_log2;
                if (key0 + i > lim) v = -__int_as_float(0x7f800000);
                sv[i] = v;
                mx = fmaxf(mx, v);
            }
        }
        const float m_new = fmaxf(m_run, mx);
        const float mref = m_new == -__int_as_float(0x7f800000) ? 0.f : m_new;
        const float alpha = ex2(m_run - mref);
        m_run = m_new;
        l_run *= alpha;
        lt_run *= alpha;
        // the previous PV must be done before O is rescaled and P overwritten
        if (j > 0 && !__syncthreads_and(mbar_wait_bounded(bar_o, (uint32_t)((j - 1) & 1), p.wait_limit_ns))) {
            failed = true;
            break;
        }
        if (j > 0) {
            tc_fence_after();
            // tile j-1's stage is free (its S and PV are done): refill it with tile j+1
            if (tid == 0 && j + 1 < n_tiles) issue(j + 1, (j + 1) & 1);
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
                tc_ld32(tO + lane_off + (uint32_t)(cb * 32), v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= alpha;
                tc_st32(tO + lane_off + (uint32_t)(cb * 32), v);
            }
        }
        // P (bf16) into shared memory, K-major 128B-swizzled [2 key blocks][128 rows][128 B]
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p0 = ex2(sv[c * 8 + 2 * e] - mref), p1 = ex2(sv[c * 8 + 2 * e + 1] - mref);
                w[e] = pack_bf16x2(p0, p1);
                l_run += p0 + p1;
                lt_run += bf16_lo(w[e]) + bf16_hi(w[e]);
            }
            const int kb = c >> 3, cc = c & 7;
            st_shared_v4(sP + (uint32_t)(kb * kBlk + r * 128 + ((cc ^ (r & 7)) << 4)), w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_shared();
        tc_fence_before();
        __syncthreads();
        // O += P V
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc_mma_bf16(tO, tc_desc(sP + (uint32_t)(kb * kBlk + k * 32), 16, 1024),
                                tc_desc(sV(st) + (uint32_t)((kb * 64 + k * 16) * 128), (uint32_t)kBlk, 1024), kIdO,
                                j > 0 || (kb | k) != 0);
            tc_commit(bar_o);
        }
    }
    // wait for the last PV, then the epilogue: out = O / lt, lse = (m + log2 l) ln 2
    if (!failed && n_tiles > 0 &&
        !__syncthreads_and(mbar_wait_bounded(bar_o, (uint32_t)((n_tiles - 1) & 1), p.wait_limit_ns)))
        failed = true;
    if (failed) {
        if (tid == 0) atomicCAS(p.status, 0, PKV_ERR_DEVICE_TIMEOUT);
    } else {
        // tcgen05.ld is collective per warp: every lane loads, rows of the group store
        tc_fence_after();
        const bool empty = n_tiles == 0 || m_run == -__int_as_float(0x7f800000);
        const float inv = empty ? 0.f : 1.f / lt_run;
        uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + grow * D);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
            if (n_tiles > 0) {
                tc_ld32(tO + lane_off + (uint32_t)(cb * 32), v);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            if (row_ok)
#pragma unroll
                for (int i = 0; i < 16; ++i) dst[cb * 16 + i] = pack_bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
        }
        if (row_ok && p.lse)
            p.lse[grow] = empty ? -__int_as_float(0x7f800000) : (m_run + __log2f(l_run)) * 0.693147180559945309f;
    }
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tc_dealloc(tmem, 256);
}

}  // namespace pkv
