// prefill_tc2_kernel.cuh -- several query rows per sequence on tcgen05, 256 rows per CTA.
//
// The same product as prefill_tc_kernel.cuh (a kv-head group's (token, head) rows packed
// token-major against the group's paged keys; AstrAI "CUDA Kernels", "Q Scheduling and KV
// Addressing"), with two 128-row query tiles A and B per CTA sharing every K/V tile: the
// copies a key tile costs are spread over twice the rows, which is what bounds the
// 128-row kernel (the copy engine's operation rate and the L2 traffic per score).
//   warps 0-3  softmax of tile A (thread r = row r = TMEM lane r)
//   warps 4-7  softmax of tile B
//   warp 8     MMAs (one lane issues)
//   warp 9     K copies (TMA, lane 2x + h: half h of page box x)
//   warp 10    V copies (TMA, lane x: page box x, both halves)
// Tensor memory holds S_A, S_B (128 columns each) and O_A, O_B (128 each).  P (bf16)
// replaces the first 64 columns of its S once the softmax has read S; the score MMA of
// the next key tile is issued only after the PV MMA that reads P has completed.  The
// MMA order per key tile j is PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), so the tensor cores
// compute one tile's products while the other tile's softmax runs.
// The online softmax keeps a reference maximum per row that moves only when a tile's
// maximum exceeds it by more than 2^8 (O is rescaled in tensor memory then).  O is
// normalised by the sum of the bf16-rounded probabilities it was accumulated from, the
// log-sum-exp uses the f32 sum (both sums kept with packed f32x2 adds).  The scale must
// be positive.
// Every wait is bounded; on a timeout the status word is set and every warp stops after
// its copies and MMAs in flight have finished.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pkv.h"
#include "prefill_tc_kernel.cuh"
#include "ptx.cuh"

namespace pkv {

constexpr int kTc2Rows = 256;      // rows per CTA: two 128-row tiles
constexpr int kTc2Threads = 352;   // 8 softmax warps, the MMA warp, the K and V copy warps
constexpr int kTc2KStages = 2;
constexpr int kTc2VStages = 3;
constexpr int kTc2PageRing = 8;

// Shared memory (bytes from a 1024-aligned base).
struct Tc2Smem {
    static constexpr int kTile = 128 * 128 * 2;              // 128 rows x 128 dims bf16, 2 column blocks
    static constexpr int q = 0;                              // Q tile t at q + t * kTile
    static constexpr int k = 2 * kTile;                      // K stage s at k + s * kTile
    static constexpr int v = k + kTc2KStages * kTile;        // V stage s at v + s * kTile
    static constexpr int bars = v + kTc2VStages * kTile;     // 32 mbarriers
    static constexpr int pages = bars + 32 * 8;              // [kTc2PageRing][16] page id of each box, -1: none
    static constexpr int tmem_slot = pages + kTc2PageRing * 16 * 4;
    static constexpr int total = tmem_slot + 16;
    static constexpr int dynamic = total;                    // the dynamic shared memory starts 1024-aligned
};
static_assert(Tc2Smem::dynamic <= 232448, "prefill_tc2_kernel: shared memory above the per-block limit");

__global__ void __launch_bounds__(kTc2Threads, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const PrefillTcParams p)
{
    constexpr int D = 128;
    constexpr int kTile = Tc2Smem::kTile;
    constexpr int kBlk = 128 * 128;      // bytes of one 64-column block of a tile
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleGap = 8.f;   // move the reference maximum only past 2^8
    // a sequence's last query tiles (the longest under the causal mask) are launched first
    const int kvh = (int)(blockIdx.x % (unsigned)p.Hkv), qp = p.q_tiles - 1 - (int)(blockIdx.x / (unsigned)p.Hkv);
    const int split = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool softmax_warp = warp < 8;
    const int qx = warp >> 2;            // the softmax warp's query tile (0: A, 1: B)
    const int G = p.G;

    if (tid == 0) {
        prefetch_tensor_map(&tmK);
        prefetch_tensor_map(&tmV);
    }
    griddep_wait();

    const int q_base = p.qo_indptr[b];
    const int n_q = p.qo_indptr[b + 1] - q_base;
    if (q_base < 0 || n_q < 0 || n_q > p.max_q_len || q_base + n_q > p.total_q) {
        if (tid == 0 && kvh == 0 && qp == 0) atomicCAS(p.status, 0, PKV_ERR_BAD_QO_INDPTR);
        return;
    }
    const int row0 = qp * kTc2Rows;
    const int nrows = min(kTc2Rows, n_q * G - row0);  // rows of the CTA (tile B may have none)
    if (nrows <= 0) return;
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_pages * p.P) {
        if (tid == 0 && kvh == 0 && qp == 0) atomicCAS(p.status, 0, PKV_ERR_BAD_SEQ_LEN);
        L = 0;
    }
    // a softmax thread's row (tile qx, lane r): token, head, global row, last key it may see
    const int r = tid & 127;
    const int crow = qx * 128 + r;       // row within the CTA
    const bool row_ok = softmax_warp && crow < nrows;
    const int tok = (row0 + (row_ok ? crow : 0)) / G, head = (row0 + (row_ok ? crow : 0)) % G;
    const size_t grow = (size_t)(q_base + tok) * p.Hq + kvh * G + head;
    const int klim = !row_ok ? -1 : (p.causal ? L - n_q + tok : L - 1);
    const int last_tok = (row0 + nrows - 1) / G;
    const int n_keys = max(0, p.causal ? min(L, L - n_q + last_tok + 1) : L);
    // key tiles of the group, split into chunks of chunk_tiles; this CTA takes chunk `split`
    // (tiles t0 .. t0 + n_tiles - 1); a group with no key tile is handled by split 0
    const int g_tiles = (n_keys + kTcKeys - 1) / kTcKeys;
    const int n_chunks = (g_tiles + p.chunk_tiles - 1) / p.chunk_tiles;
    if (split >= max(n_chunks, 1)) return;
    const int t0 = split * p.chunk_tiles;
    const int n_tiles = min(p.chunk_tiles, g_tiles - t0);
    const bool direct = n_chunks <= 1;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_addr(smem_raw);
    if (base & 1023u) {  // the swizzled tiles need a 1024-aligned base
        if (tid == 0) atomicCAS(p.status, 0, PKV_ERR_UNSUPPORTED);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + Tc2Smem::bars);
    int *sm_pg = reinterpret_cast<int *>(smem_raw + Tc2Smem::pages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + Tc2Smem::tmem_slot);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    constexpr int kKFull = 0, kKEmpty = kKFull + kTc2KStages, kVFull = kKEmpty + kTc2KStages,
                  kVEmpty = kVFull + kTc2VStages, kSFull = kVEmpty + kTc2VStages, kPFull = kSFull + 2,
                  kODone = kPFull + 2, kDrain = kODone + 2, kQFull = kDrain + 1;
    static_assert(kQFull < 32, "prefill_tc2_kernel: more mbarriers than the shared-memory slots");
    auto k_full = [&](int s) { return bar(kKFull + s); };
    auto k_empty = [&](int s) { return bar(kKEmpty + s); };
    auto v_full = [&](int s) { return bar(kVFull + s); };
    auto v_empty = [&](int s) { return bar(kVEmpty + s); };
    auto s_full = [&](int x) { return bar(kSFull + x); };   // per query tile
    auto p_full = [&](int x) { return bar(kPFull + x); };
    auto o_done = [&](int x) { return bar(kODone + x); };
    const uint32_t drain = bar(kDrain), q_full = bar(kQFull);
    auto sQ = [&](int x) { return base + Tc2Smem::q + (uint32_t)(x * kTile); };
    auto sK = [&](int s) { return base + Tc2Smem::k + (uint32_t)(s * kTile); };
    auto sV = [&](int s) { return base + Tc2Smem::v + (uint32_t)(s * kTile); };

    if (tid == 0) {
        for (int s = 0; s < kTc2KStages; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < kTc2VStages; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(s_full(x), 2);  // the MMA's commit + the issuing lane (publishes the tile's page ids)
            mbar_init(p_full(x), 4);
            mbar_init(o_done(x), 1);
        }
        mbar_init(drain, 1);
        mbar_init(q_full, 8);  // one arrival per softmax warp once its Q rows are in shared memory
        fence_barrier_init();
    }
    // TMEM columns: S_A 0..127, S_B 128..255, O_A 256..383, O_B 384..511; P_x in S_x 0..63
    if (warp == 0) tc_alloc(smem_addr(tmem_slot), 512);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto tS = [&](int x) { return tmem + (uint32_t)(x * 128); };
    auto tO = [&](int x) { return tmem + 256u + (uint32_t)(x * 128); };
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int log2box = p.log2P < 7 ? p.log2P : 7;
    const int box_t = 1 << log2box;
    const int nbox = kTcKeys / box_t;
    bool failed = false;

    if (warp >= 9 && n_tiles > 0) {
        // ---- copy warps: warp 9 streams K (lane 2x + h: half h of page box x), warp 10 V
        // (lane x: page box x, both halves); the block-table entry is read a tile early
        const bool is_k = warp == 9;
        const int stages = is_k ? kTc2KStages : kTc2VStages;
        const uint64_t policy = l2_policy_evict_first();
        const int x = is_k ? lane >> 1 : lane, dc = is_k ? lane & 1 : 0;
        auto fetch = [&](int j) {
            const int key = (t0 + j) * kTcKeys + x * box_t;
            return (dc == 0 && x < nbox && j < n_tiles && key < n_keys)
                       ? p.block_table[(size_t)b * p.max_pages + (key >> p.log2P)]
                       : -1;
        };
        int raw = fetch(0);
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % stages;
            const int next_raw = fetch(j + 1);
            const bool has_key = x < nbox && (t0 + j) * kTcKeys + x * box_t < n_keys;
            const int pg_raw = is_k ? __shfl_sync(0xffffffffu, raw, lane & ~1) : raw;
            const int pg = has_key && (unsigned)pg_raw < (unsigned)p.num_pages ? pg_raw : -1;
            if (is_k && dc == 0 && has_key && pg < 0) atomicCAS(p.status, 0, PKV_ERR_BAD_PAGE_INDEX);
            const uint32_t ok = __ballot_sync(0xffffffffu, pg >= 0);  // one bit per copy
            if (j >= stages) {
                const uint32_t empty = is_k ? k_empty(st) : v_empty(st);
                if (!__all_sync(0xffffffffu,
                                mbar_wait_bounded(empty, (uint32_t)((j / stages - 1) & 1), p.wait_limit_ns))) {
                    failed = true;
                    break;
                }
            }
            if (is_k) {  // publish the tile's page ids (read by the softmax and the MMA warp)
                if (dc == 0 && x < nbox) sm_pg[(j % kTc2PageRing) * 16 + x] = pg;
                __syncwarp();
            }
            const uint32_t full = is_k ? k_full(st) : v_full(st);
            const uint32_t copy_bytes = (uint32_t)box_t * (is_k ? 128u : 256u);
            if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)__popc(ok) * copy_bytes);
            __syncwarp();
            if (pg >= 0) {
                const int row = pg * p.P + (((t0 + j) * kTcKeys + x * box_t) & (p.P - 1));
                if (is_k)
                    tma_load_3d(sK(st) + (uint32_t)(dc * kBlk + x * box_t * 128), &tmK, dc * 64, kvh, row, full,
                                policy);
                else
                    tma_load_4d(sV(st) + (uint32_t)(x * box_t * 256), &tmV, 0, row, 0, kvh, full, policy);
            }
            issued = j + 1;
            raw = next_raw;
        }
        // the last copies have landed before the CTA exits (consumed, or waited for here)
        for (int t = max(0, issued - stages); t < issued; ++t)
            mbar_wait_bounded(is_k ? k_full(t % stages) : v_full(t % stages), (uint32_t)((t / stages) & 1),
                              p.wait_limit_ns);
    } else if (warp == 8 && n_tiles > 0) {
        // ---- MMA warp: every lane waits, lane 0 issues
        const bool leader = lane == 0;
        auto wait_all = [&](uint32_t bar_addr, int parity) {
            return __all_sync(0xffffffffu, mbar_wait_bounded(bar_addr, (uint32_t)(parity & 1), p.wait_limit_ns));
        };
        // zeroes the V rows of tile j whose keys are invalid (past n_keys, bad page): key k
        // is row k % box_t of box k / box_t, 2 halves x 8 chunks of 16 bytes; lanes 0-15
        // clear the even keys, 16-31 the odd ones, lane & 15 naming the chunk
        auto zero_invalid_v = [&](int j) {
            const int *ids = sm_pg + (j % kTc2PageRing) * 16;
            const int first_past = min(kTcKeys, max(0, n_keys - (t0 + j) * kTcKeys));  // keys past n_keys: [first_past, 128)
            bool bad = false;  // a missing page among the keys before that
            for (int bx = 0; bx < nbox; ++bx) bad |= ids[bx] < 0 && (bx << log2box) < first_past;
            if (first_past == kTcKeys && !bad) return;
            const uint32_t dst = sV(j % kTc2VStages) + (uint32_t)(((lane >> 3) & 1) * box_t * 128 + (lane & 7) * 16);
            auto zero_key = [&](int k) {
                st_shared_v4(dst + (uint32_t)((k >> log2box) * box_t * 256 + (k & (box_t - 1)) * 128), 0u, 0u, 0u, 0u);
            };
            for (int k = first_past + (lane >> 4); k < kTcKeys; k += 2) zero_key(k);
            if (bad)
                for (int bx = 0; bx < nbox; ++bx)
                    if (ids[bx] < 0 && (bx << log2box) < first_past)
                        for (int k = (bx << log2box) + (lane >> 4); k < min((bx + 1) << log2box, first_past); k += 2)
                            zero_key(k);
            fence_proxy_async_shared();
            __syncwarp();
        };
        // V operand of the 16-key MMA step kk: 8-key groups 1024 bytes apart within a box
        // (the 64-dim halves box_t * 128 apart), or, with 8-key boxes, one box per group
        auto v_desc = [&](uint32_t stage, int kk) {
            const int k0 = kk * 16;
            return box_t == 8 ? tc_desc(stage + (uint32_t)(kk * 4096), 1024, 2048)
                              : tc_desc(stage + (uint32_t)((k0 >> log2box) * box_t * 256 + (k0 & (box_t - 1)) * 128),
                                        (uint32_t)(box_t * 128), 1024);
        };
        constexpr uint32_t kIdS = tc_idesc_bf16(128, kTcKeys, false);
        constexpr uint32_t kIdO = tc_idesc_bf16(128, D, true);
        auto issue_s = [&](int x, int j) {  // S_x = Q_x K(j)^T
            if (leader) {
                const uint32_t kst = sK(j % kTc2KStages);
                tc_fence_after();
#pragma unroll
                for (int dcb = 0; dcb < 2; ++dcb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma_bf16(tS(x), tc_desc(sQ(x) + (uint32_t)(dcb * kBlk + k * 32), 16, 1024),
                                    tc_desc(kst + (uint32_t)(dcb * kBlk + k * 32), 16, 1024), kIdS, (dcb | k) != 0);
                tc_commit(s_full(x));
                if (x == 1) tc_commit(k_empty(j % kTc2KStages));  // both tiles' scores have read K(j)
                mbar_arrive(s_full(x));
            }
            __syncwarp();
        };
        auto issue_pv = [&](int x, int j) {  // O_x += P_x V(j), P_x in the first 64 columns of S_x
            if (leader) {
                const uint32_t vst = sV(j % kTc2VStages);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_bf16_ts(tO(x), tS(x) + (uint32_t)(kk * 8), v_desc(vst, kk), kIdO, j > 0 || kk > 0);
                tc_commit(o_done(x));
                if (x == 1) tc_commit(v_empty(j % kTc2VStages));  // both tiles' PV have read V(j)
            }
            __syncwarp();
        };
        if (wait_all(q_full, 0) && wait_all(k_full(0), 0)) {
            issue_s(0, 0);
            issue_s(1, 0);
        } else {
            failed = true;
        }
        for (int j = 0; j < n_tiles && !failed; ++j) {
            if (!wait_all(v_full(j % kTc2VStages), j / kTc2VStages)) {
                failed = true;
                break;
            }
            zero_invalid_v(j);
            for (int x = 0; x < 2 && !failed; ++x) {
                if (!wait_all(p_full(x), j)) {
                    failed = true;
                    break;
                }
                issue_pv(x, j);
                if (j + 1 < n_tiles) {
                    // S_x(j+1) overwrites the columns PV_x(j) reads P_x from; MMAs issued by one
                    // thread execute in issue order, so it follows PV_x(j) without a wait
                    if (x == 0 && !wait_all(k_full((j + 1) % kTc2KStages), (j + 1) / kTc2KStages)) {
                        failed = true;
                        break;
                    }
                    issue_s(x, j + 1);
                }
            }
        }
        // the MMAs in flight finish before the CTA exits
        if (leader) {
            tc_commit(drain);
            if (!mbar_wait_bounded(drain, 0, p.wait_limit_ns)) failed = true;
        }
    } else if (softmax_warp && n_tiles > 0) {
        // ---- softmax warps of tile qx: thread r owns row r.  Q rows into shared memory first
        // (128B-swizzled [2 column blocks][128 rows][128 B] per tile), while the copies start.
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + grow * D);
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const uint4 v = row_ok ? __ldg(src + cq) : make_uint4(0u, 0u, 0u, 0u);
                const int dc = cq >> 3, cc = cq & 7;
                st_shared_v4(sQ(qx) + (uint32_t)(dc * kBlk + r * 128 + ((cc ^ (r & 7)) << 4)), v.x, v.y, v.z, v.w);
            }
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        const float c = p.scale_log2;  // > 0
        float m_ref = kNegInf, l_run = 0.f, lt_run = 0.f;
        const int row_lim = min(n_keys, klim + 1);  // keys [0, row_lim) are visible to this row
        for (int j = 0; j < n_tiles; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full(qx), (uint32_t)(j & 1), p.wait_limit_ns))) {
                failed = true;
                break;
            }
            tc_fence_after();
            uint32_t sr[kTcKeys];
            tc_ld128(tS(qx) + lane_off, sr);
            // masking: none on tiles every row of the warp sees whole, the row's limit on
            // the diagonal, a key bitmask where a page is missing
            const int *ids = sm_pg + (j % kTc2PageRing) * 16;
            bool pages_ok = true;
            for (int bx = 0; bx < nbox; ++bx) pages_ok &= ids[bx] >= 0;
            const int lim = row_lim - (t0 + j) * kTcKeys;
            if (!pages_ok) {
                uint32_t okw[4] = {0u, 0u, 0u, 0u};
                for (int bx = 0; bx < nbox; ++bx) {
                    if (ids[bx] < 0) continue;
                    const int k0 = bx << log2box, k1 = k0 + box_t;
                    for (int w = k0 >> 5; w < ((k1 + 31) >> 5); ++w) {
                        const int lo = max(k0, 32 * w) - 32 * w, n = min(k1, 32 * w + 32) - 32 * w - lo;
                        okw[w] |= (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << lo;
                    }
                }
#pragma unroll
                for (int i = 0; i < kTcKeys; ++i)
                    if (!((okw[i >> 5] >> (i & 31)) & 1u) || i >= lim) sr[i] = 0xff800000u;  // -inf
            } else if (__any_sync(0xffffffffu, lim < kTcKeys)) {
#pragma unroll
                for (int i = 0; i < kTcKeys; ++i)
                    if (i >= lim) sr[i] = 0xff800000u;
            }
            // tile maximum of the unscaled scores: eight chains of three-input max
            float mx8[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) mx8[a] = __uint_as_float(sr[a]);
#pragma unroll
            for (int i = 8; i < kTcKeys; i += 16)
#pragma unroll
                for (int a = 0; a < 8; ++a)
                    mx8[a] = i + 8 + a < kTcKeys
                                 ? fmax3(mx8[a], __uint_as_float(sr[i + a]), __uint_as_float(sr[i + 8 + a]))
                                 : fmaxf(mx8[a], __uint_as_float(sr[i + a]));
            const float mx =
                fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], fmax3(mx8[5], mx8[6], mx8[7]))) * c;
            // reference maximum: set at the first visible key, moved only past a 2^8 rise
            float alpha = 1.f;
            if (mx != kNegInf && (m_ref == kNegInf || mx > m_ref + kRescaleGap)) {
                alpha = m_ref == kNegInf ? 0.f : ex2(m_ref - mx);
                m_ref = mx;
                l_run *= alpha;
                lt_run *= alpha;
            }
            // PV(j-1) completed before S(j) was issued: O may be rescaled now
            if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tc_ld32(tO(qx) + lane_off + (uint32_t)(cb * 32), v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tc_st32(tO(qx) + lane_off + (uint32_t)(cb * 32), v);
                }
            }
            const float neg_ref = m_ref == kNegInf ? 0.f : -m_ref;
            // p = 2^(s c - m) for two keys at a time (packed f32 pairs for the FMA and the sums)
            const uint64_t c2 = f32x2(c, c), nr2 = f32x2(neg_ref, neg_ref);
            uint64_t ls2[2] = {0ull, 0ull};
            float lta[2] = {0.f, 0.f}, ltb[2] = {0.f, 0.f};  // the bf16 sums: low and high halves
            uint32_t pw[kTcKeys / 2];
#pragma unroll
            for (int i = 0; i < kTcKeys / 2; ++i) {
                float a0, a1;
                f32x2_split(fma_f32x2(f32x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])), c2, nr2), a0,
                            a1);
                const float p0 = ex2(a0), p1 = ex2(a1);
                pw[i] = pack_bf16x2(p0, p1);
                ls2[i & 1] = add_f32x2(ls2[i & 1], f32x2(p0, p1));
                add_bf16x2_to_f32(pw[i], lta[i & 1], ltb[i & 1]);
            }
            {
                float l0, l1, l2, l3;
                f32x2_split(ls2[0], l0, l1);
                f32x2_split(ls2[1], l2, l3);
                l_run += (l0 + l1) + (l2 + l3);
                lt_run += (lta[0] + ltb[0]) + (lta[1] + ltb[1]);
            }
            // P (bf16 pairs) into the first 64 columns of this row's S lane
            tc_st64(tS(qx) + lane_off, pw);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(qx));
        }
        // epilogue: out = O / lt, lse = (m + log2 l) ln 2
        if (!failed && !__all_sync(0xffffffffu, mbar_wait_bounded(o_done(qx), (uint32_t)((n_tiles - 1) & 1),
                                                                   p.wait_limit_ns)))
            failed = true;
        if (!failed) {
            tc_fence_after();
            const bool empty = m_ref == kNegInf;
            const float inv = empty ? 0.f : 1.f / lt_run;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + grow * D);
            const float row_lse = empty ? kNegInf : (m_ref + __log2f(l_run)) * 0.693147180559945309f;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
                tc_ld32(tO(qx) + lane_off + (uint32_t)(cb * 32), v);  // collective: every lane loads
                if (row_ok && direct) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[cb * 4 + i] = make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                                     pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                                     pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                                     pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
                } else if (row_ok) {
                    tc_store_partial(p, split, grow, cb, v, inv);
                }
            }
            if (row_ok && direct && p.lse) p.lse[grow] = row_lse;
            if (row_ok && !direct) p.part_lse[split * p.total_rows + grow] = row_lse;
        }
    }
    if (softmax_warp && n_tiles == 0 && row_ok) {  // no key visible to the CTA: out = 0, lse = -inf
        uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + grow * D);
        for (int i = 0; i < D / 2; ++i) dst[i] = 0u;
        if (p.lse) p.lse[grow] = kNegInf;
    }
    if (failed) atomicCAS(p.status, 0, PKV_ERR_DEVICE_TIMEOUT);
    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, 512);
    }
    if (!direct) {  // the group's last split to finish merges the partials (also after a timeout,
                    // so the counter returns to 0 for the next call)
        int *last = reinterpret_cast<int *>(smem_raw + Tc2Smem::tmem_slot + 4);
        __threadfence();
        __syncthreads();
        if (tid == 0)
            *last = atomicInc(reinterpret_cast<unsigned *>(p.counters + ((size_t)b * p.q_tiles + qp) * p.Hkv + kvh),
                              (unsigned)(n_chunks - 1)) == (unsigned)(n_chunks - 1);
        __syncthreads();
        if (*last) {  // every warp merges rows warp, warp + W, ... of this CTA
            __threadfence();
            for (int cr = warp; cr < nrows; cr += kTc2Threads / 32) {
                const int rt = (row0 + cr) / G, rh = (row0 + cr) % G;
                tc_merge_row_warp(p, n_chunks, (size_t)(q_base + rt) * p.Hq + kvh * G + rh, lane);
            }
        }
    }
}

}  // namespace pkv
