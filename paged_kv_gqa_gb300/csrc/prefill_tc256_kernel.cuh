// prefill_tc256_kernel.cuh -- several query rows per sequence on tcgen05 at head dim 256.
//
// The 128-row design of prefill_tc_kernel.cuh (a kv-head group's (token, head) rows packed
// token-major against the group's paged keys; AstrAI "CUDA Kernels", "Q Scheduling and KV
// Addressing") for D = 256, on a bf16 cache or (KV8) an fp8 one.  The tiles are 64 keys instead of 128, so that Q
// (128 rows x 256 dims), two K stages and two V stages of 64 keys x 256 dims fit in shared
// memory, and S, O (256 columns) and the row sums fit in tensor memory:
//   warps 0-3  softmax (thread r = row r = TMEM lane r)
//   warp 4     MMAs (one lane issues)
//   warp 5     K copies (TMA, lane 4x + h: 64-dim block h of page box x)
//   warp 6     V copies (TMA, lane x: page box x, all four 64-dim blocks)
//   warps 7-10 (fp8 only) converters: the codes and scales warps 5-6 stage, dequantised to bf16
//              tiles in the layout the bf16 copies land
// S = Q K^T: M = 128 rows, N = 64 keys, K = 256 (sixteen 16-deep MMAs, Q and K K-major,
// 128B-swizzled); O += P V: N = 256 dims, K = 64 keys (P from tensor memory, V read MN-major
// in the layout one copy per page box lands: [box][4 dim blocks][keys][64]); the row sums of
// the bf16-rounded P on the tensor cores too (P x a tile of ones).  S is double-buffered, so
// the score MMA of the next tile runs while the softmax reads the current one.  The online
// softmax keeps a reference maximum that moves only past a 2^8 rise (O rescaled in tensor
// memory then); O is normalised by the sum of the bf16-rounded probabilities, the lse uses
// the f32 sum.  The scale must be positive.  Keys past the last one the CTA's rows may see,
// or in a page whose id is out of range, are masked in the scores and zeroed in V's rows.
// Every wait is bounded; on a timeout the status word is set, the issuing lane waits
// (bounded) for its copies and MMAs in flight, and every warp stops.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pkv.h"
#include "prefill_tc_kernel.cuh"
#include "ptx.cuh"

namespace pkv {

constexpr int kT256Keys = 64;        // keys per tile

// Per cache type: threads, bf16 K and V stages, fp8 staging stages.  bf16: 4 softmax warps,
// the MMA warp, the K and V copy warps; K and V land by TMA straight into two stages each.
// fp8: the copy warps land the e4m3 codes and scales in two staging stages, and two K and two
// V converter warps (7-8, 9-10) write them, dequantised to bf16, into one K and one V stage in
// the layout the bf16 copies land (two bf16 stages each do not fit beside the staging).
template <bool KV8>
struct T256Cfg {
    static constexpr int threads = KV8 ? 352 : 224;
    static constexpr int k_stages = KV8 ? 1 : 2;
    static constexpr int v_stages = KV8 ? 1 : 2;
    static constexpr int s8_stages = KV8 ? 2 : 0;
};
constexpr int kT256Threads = T256Cfg<false>::threads;
constexpr int kT2568Threads = T256Cfg<true>::threads;
constexpr int kT256KStages = T256Cfg<false>::k_stages;

// Shared memory (bytes from a 1024-aligned base).
template <bool KV8>
struct T256SmemT {
    static constexpr int kQBlk = kTcRows * 128;                  // one 64-dim block of Q: 128 rows x 128 B
    static constexpr int kKBlk = kT256Keys * 128;                // one 64-dim block of a K tile: 64 keys x 128 B
    static constexpr int kStage = kT256Keys * 256 * 2;           // a K or V tile: 64 keys x 256 dims bf16
    static constexpr int kCodes = kT256Keys * 256;               // 64 keys x 256 e4m3 codes
    static constexpr int q = 0;                                  // [4 blocks][128 rows][128 B]
    static constexpr int k = 4 * kQBlk;                          // K stage s at k + s * kStage: [4][64][128 B]
    static constexpr int v = k + T256Cfg<KV8>::k_stages * kStage;  // V stage s: [box][4][box keys][128 B]
    static constexpr int ones = v + T256Cfg<KV8>::v_stages * kStage;  // 16 x 64 bf16 ones, the row-sum MMA's B
    // fp8 staging stage s at s8 + s * 2 kCodes: [K codes][V codes], each as the page boxes land
    // ([box][2 blocks of 128 codes][box keys][128 B], 128B-swizzled); its scales at sc8 + s * 512:
    // [K 64][V 64] f32
    static constexpr int s8 = (ones + 2048 + 1023) / 1024 * 1024;
    static constexpr int sc8 = s8 + T256Cfg<KV8>::s8_stages * 2 * kCodes;
    static constexpr int bars = sc8 + T256Cfg<KV8>::s8_stages * 2 * kT256Keys * 4;  // 32 mbarriers
    static constexpr int pages = bars + 32 * 8;                  // [kTcPageRing][16] page id of each box, -1: none
    static constexpr int tmem_slot = pages + kTcPageRing * 16 * 4;
    static constexpr int total = tmem_slot + 16;
    static constexpr int dynamic = total;                        // the dynamic shared memory starts 1024-aligned
};
using T256Smem = T256SmemT<false>;
using T2568Smem = T256SmemT<true>;
static_assert(T256Smem::dynamic <= 232448 && T2568Smem::dynamic <= 232448,
              "prefill_tc256_kernel: shared memory above the per-block limit");
static_assert(T256Smem::ones % 1024 == 0 && T2568Smem::ones % 1024 == 0,
              "prefill_tc256_kernel: tiles must stay 1024-aligned");

// A split's row result into the partials (O / lt in f32); o holds dims 32 cb .. 32 cb + 31 of
// a 256-dim row.
__device__ __forceinline__ void t256_store_partial(const PrefillTcParams &p, int c, size_t grow, int cb,
                                                   const float (&o)[32], float inv)
{
    float4 *dst = reinterpret_cast<float4 *>(p.part_out + (c * p.total_rows + grow) * 256) + cb * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
}

// The merge of tc_merge_row_warp for a 256-dim row: lane l owns dims 4l .. 4l + 3 and
// 128 + 4l .. 128 + 4l + 3, the splits combined in split order with the same weights.
__device__ __forceinline__ void t256_merge_row_warp(const PrefillTcParams &p, int n_chunks, size_t grow, int lane)
{
    constexpr float kLog2e = 1.4426950408889634074f;
    const float ninf = __int_as_float(0xff800000);
    float m = ninf;
    for (int c = lane; c < n_chunks; c += 32) m = fmaxf(m, __ldcg(p.part_lse + c * p.total_rows + grow));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float mr = m == ninf ? 0.f : m;
    float wsum = 0.f;
    for (int c = lane; c < n_chunks; c += 32) wsum += ex2((__ldcg(p.part_lse + c * p.total_rows + grow) - mr) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = m == ninf ? 0.f : 1.f / wsum;
    float4 a[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int c0 = 0; c0 < n_chunks; c0 += 32) {
        // weight of split c0 + lane, broadcast below
        const float wl = c0 + lane < n_chunks
                             ? ex2((__ldcg(p.part_lse + (c0 + lane) * p.total_rows + grow) - mr) * kLog2e) * inv
                             : 0.f;
        const int nc = min(32, n_chunks - c0);
        for (int k0 = 0; k0 < nc; k0 += 4) {
            float4 v[4][2];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    v[k][hh] = k0 + k < nc ? __ldcg(reinterpret_cast<const float4 *>(
                                                        p.part_out + ((size_t)(c0 + k0 + k) * p.total_rows + grow) * 256) +
                                                    hh * 32 + lane)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, (k0 + k) & 31);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    a[hh].x += v[k][hh].x * w;
                    a[hh].y += v[k][hh].y * w;
                    a[hh].z += v[k][hh].z * w;
                    a[hh].w += v[k][hh].w * w;
                }
            }
        }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
        reinterpret_cast<uint2 *>(p.out + grow * 256)[hh * 32 + lane] =
            make_uint2(pack_bf16x2(a[hh].x, a[hh].y), pack_bf16x2(a[hh].z, a[hh].w));
    if (lane == 0 && p.lse) p.lse[grow] = m == ninf ? ninf : m + __logf(wsum);
}

template <bool KV8>
__global__ void __launch_bounds__(T256Cfg<KV8>::threads, 1)
    prefill_tc256_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const PrefillTcParams p)
{
    using Smem = T256SmemT<KV8>;
    constexpr int D = 256;
    constexpr int KT = kT256Keys;
    constexpr int kThreads = T256Cfg<KV8>::threads;
    constexpr int kKStages = T256Cfg<KV8>::k_stages, kVStages = T256Cfg<KV8>::v_stages;
    constexpr int kS8Stages = T256Cfg<KV8>::s8_stages;
    constexpr int kS8Div = kS8Stages > 0 ? kS8Stages : 1;  // the bf16 instantiation compiles the fp8 roles too
    constexpr int kQBlk = Smem::kQBlk, kKBlk = Smem::kKBlk, kStage = Smem::kStage, kCodes = Smem::kCodes;
    const float kNegInf = __int_as_float(0xff800000);
    constexpr float kRescaleGap = 8.f;   // move the reference maximum only past 2^8
    // a sequence's last query tiles (the longest under the causal mask) are launched first
    const int kvh = (int)(blockIdx.x % (unsigned)p.Hkv), qt = p.q_tiles - 1 - (int)(blockIdx.x / (unsigned)p.Hkv);
    const int split = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer_warp = warp >= 4;  // the MMA warp and the copy warps
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
    // a softmax thread's row: token, head, global row, last key it may see
    const int r = tid & 127;
    const bool row_ok = !issuer_warp && r < nrows;
    const int tok = (row0 + (row_ok ? r : 0)) / G, head = (row0 + (row_ok ? r : 0)) % G;
    const size_t grow = (size_t)(q_base + tok) * p.Hq + kvh * G + head;
    const int klim = !row_ok ? -1 : (p.causal ? L - n_q + tok : L - 1);
    // keys any row of the CTA may see
    const int last_tok = (row0 + nrows - 1) / G;
    const int n_keys = max(0, p.causal ? min(L, L - n_q + last_tok + 1) : L);
    // key tiles of the group, split into chunks of chunk_tiles; this CTA takes chunk `split`
    // (tiles t0 .. t0 + n_tiles - 1); a group with no key tile is handled by split 0
    const int g_tiles = (n_keys + KT - 1) / KT;
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
    const uint32_t sQ = base + Smem::q, sOnes = base + Smem::ones;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + Smem::bars);
    int *sm_pg = reinterpret_cast<int *>(smem_raw + Smem::pages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + Smem::tmem_slot);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    constexpr int kKFull = 0, kKEmpty = kKFull + kKStages, kVFull = kKEmpty + kKStages,
                  kVEmpty = kVFull + kVStages, kSFull = kVEmpty + kVStages, kSFree = kSFull + 2,
                  kPFull = kSFree + 2, kODone = kPFull + 1, kDrain = kODone + 1, kQFull = kDrain + 1,
                  kK8Full = kQFull + 1, kK8Empty = kK8Full + kS8Stages, kV8Full = kK8Empty + kS8Stages,
                  kV8Empty = kV8Full + kS8Stages, kBarEnd = kV8Empty + kS8Stages;
    static_assert(kBarEnd <= 32, "prefill_tc256_kernel: more mbarriers than the shared-memory slots");
    auto k_full = [&](int s) { return bar(kKFull + s); };
    auto k_empty = [&](int s) { return bar(kKEmpty + s); };
    auto v_full = [&](int s) { return bar(kVFull + s); };
    auto v_empty = [&](int s) { return bar(kVEmpty + s); };
    auto k8_full = [&](int s) { return bar(kK8Full + s); };    // fp8: codes and scales of a staging stage landed
    auto k8_empty = [&](int s) { return bar(kK8Empty + s); };  // fp8: the converters have read the stage
    auto v8_full = [&](int s) { return bar(kV8Full + s); };
    auto v8_empty = [&](int s) { return bar(kV8Empty + s); };
    auto s_full = [&](int s) { return bar(kSFull + s); };
    auto s_free = [&](int s) { return bar(kSFree + s); };
    const uint32_t p_full = bar(kPFull), o_done = bar(kODone), drain = bar(kDrain), q_full = bar(kQFull);
    auto sK = [&](int s) { return base + Smem::k + (uint32_t)(s * kStage); };
    auto sV = [&](int s) { return base + Smem::v + (uint32_t)(s * kStage); };
    auto s8 = [&](int s) { return base + Smem::s8 + (uint32_t)(s * 2 * kCodes); };       // fp8 staging codes
    auto sc8 = [&](int s) { return base + Smem::sc8 + (uint32_t)(s * 2 * KT * 4); };     // fp8 staging scales

    if (tid == 0) {
        // bf16: a full K/V stage is the copy lane's expect_tx; fp8: one arrival per converter warp
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(k_full(s), KV8 ? 2 : 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(v_full(s), KV8 ? 2 : 1);
            mbar_init(v_empty(s), 1);
        }
        for (int s = 0; s < kS8Stages; ++s) {
            mbar_init(k8_full(s), 1);
            mbar_init(k8_empty(s), 2);
            mbar_init(v8_full(s), 1);
            mbar_init(v8_empty(s), 2);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(s_full(s), 2);  // the MMA's commit + the issuing lane (publishes the tile's page ids)
            mbar_init(s_free(s), 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        mbar_init(q_full, 4);  // one arrival per softmax warp once its Q rows are in shared memory
        fence_barrier_init();
    }
    // TMEM columns: S0 0..63, S1 64..127, O 128..383, the row sums of bf16 P 384..399,
    // P (bf16 pairs) 448..479
    if (warp == 0) tc_alloc(smem_addr(tmem_slot), 512);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + 128u, tL = tmem + 384u, tP = tmem + 448u;
    auto tS = [&](int sb) { return tmem + (uint32_t)(sb * KT); };
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int log2box = p.log2P < 6 ? p.log2P : 6;
    const int box_t = 1 << log2box;    // keys per page box: min(P, 64)
    const int nbox = KT / box_t;       // 1 .. 8
    bool failed = false;

    if (KV8 && warp >= 7 && n_tiles > 0) {
        // ---- fp8 converter warps: 7-8 write K tiles, 9-10 V tiles.  A task is 16 codes (one
        // 16-byte chunk of a key row): read from the staging box (128B-swizzled), scaled to bf16,
        // and stored as the two 16-byte chunks the bf16 copies would land
        const bool is_k = warp < 9;
        const int ct = (warp - (is_k ? 7 : 9)) * 32 + lane;  // 0..63
        for (int j = 0; j < n_tiles; ++j) {
            const int st8 = j % kS8Div;
            const bool ok = mbar_wait_bounded(is_k ? k8_full(st8) : v8_full(st8), (uint32_t)((j / kS8Div) & 1),
                                              p.wait_limit_ns) &&
                            (is_k ? (j < kKStages || mbar_wait_bounded(k_empty(j % kKStages),
                                                                        (uint32_t)((j / kKStages - 1) & 1),
                                                                        p.wait_limit_ns))
                                  : (j < kVStages || mbar_wait_bounded(v_empty(j % kVStages),
                                                                        (uint32_t)((j / kVStages - 1) & 1),
                                                                        p.wait_limit_ns)));
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                break;
            }
            const uint32_t src = s8(st8) + (is_k ? 0u : (uint32_t)kCodes);
            const uint32_t scl = sc8(st8) + (is_k ? 0u : (uint32_t)(KT * 4));
            const uint32_t dst = is_k ? sK(j % kKStages) : sV(j % kVStages);
#pragma unroll 4
            for (int t = ct; t < KT * 16; t += 64) {
                const int key = t >> 4, ch = t & 15;
                const int bx = key >> log2box, r = key & (box_t - 1);
                // codes: [box][2 blocks of 128][box keys][128 B], swizzled on the key within the box
                const uint4 c = tc_ld_shared_v4(src + (uint32_t)(bx * box_t * 256 + (ch >> 3) * box_t * 128 + r * 128 +
                                                                  (((ch & 7) ^ (r & 7)) << 4)));
                uint32_t o[8];
                e4m3x16_scaled_to_bf16(c, ld_shared_f32(scl + (uint32_t)(key * 4)), o);
                // dims 16 ch .. 16 ch + 15: 64-dim block ch / 4, chunks 2 (ch % 4) and the next.
                // K: [block][key][128 B]; V: [box][block][box key][128 B]
                const int dc = ch >> 2, c16 = (ch & 3) * 2, sw = is_k ? (key & 7) : (r & 7);
                const uint32_t row = is_k ? dst + (uint32_t)(dc * kKBlk + key * 128)
                                          : dst + (uint32_t)(bx * box_t * 512 + dc * box_t * 128 + r * 128);
                st_shared_v4(row + (uint32_t)((c16 ^ sw) << 4), o[0], o[1], o[2], o[3]);
                st_shared_v4(row + (uint32_t)(((c16 + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_shared();  // the MMAs read the tile through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(is_k ? k_full(j % kKStages) : v_full(j % kVStages));
                mbar_arrive(is_k ? k8_empty(st8) : v8_empty(st8));
            }
        }
    } else if (KV8 && (warp == 5 || warp == 6) && n_tiles > 0) {
        // ---- fp8 copy warps: warp 5 lands K codes and scales, warp 6 V's, in the staging
        // stages; lane x copies box x (box_t keys of one page: one code box, one scale run)
        const bool is_k = warp == 5;
        const uint64_t policy = l2_policy_evict_first();
        const int x = lane;
        auto fetch = [&](int j) {
            const int key = (t0 + j) * KT + x * box_t;
            return (x < nbox && j < n_tiles && key < n_keys) ? p.block_table[(size_t)b * p.max_pages + (key >> p.log2P)]
                                                            : -1;
        };
        int raw = fetch(0);
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % kS8Div;
            const int next_raw = fetch(j + 1);
            const bool has_key = x < nbox && (t0 + j) * KT + x * box_t < n_keys;
            const int pg = has_key && (unsigned)raw < (unsigned)p.num_pages ? raw : -1;
            if (is_k && has_key && pg < 0) atomicCAS(p.status, 0, PKV_ERR_BAD_PAGE_INDEX);
            const uint32_t ok = __ballot_sync(0xffffffffu, pg >= 0);
            if (j >= kS8Stages &&
                !__all_sync(0xffffffffu, mbar_wait_bounded(is_k ? k8_empty(st) : v8_empty(st),
                                                           (uint32_t)((j / kS8Div - 1) & 1), p.wait_limit_ns))) {
                failed = true;
                break;
            }
            if (is_k) {  // publish the tile's page ids (read by the softmax and the MMA warp)
                if (x < nbox) sm_pg[(j % kTcPageRing) * 16 + x] = pg;
                __syncwarp();
            }
            const uint32_t full = is_k ? k8_full(st) : v8_full(st);
            if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)__popc(ok) * (uint32_t)box_t * (256u + 4u));
            __syncwarp();
            if (pg >= 0) {
                const int slot = ((t0 + j) * KT + x * box_t) & (p.P - 1);
                tma_load_4d(s8(st) + (is_k ? 0u : (uint32_t)kCodes) + (uint32_t)(x * box_t * 256), is_k ? &tmK : &tmV,
                            0, pg * p.P + slot, 0, kvh, full, policy);
                bulk_copy_g2s(sc8(st) + (is_k ? 0u : (uint32_t)(KT * 4)) + (uint32_t)(x * box_t * 4),
                              (is_k ? p.k_scale : p.v_scale) + ((size_t)pg * p.Hkv + kvh) * p.P + slot,
                              (uint32_t)box_t * 4u, full);
            }
            issued = j + 1;
            raw = next_raw;
        }
        // the last copies have landed before the CTA exits (consumed, or waited for here)
        for (int t = max(0, issued - kS8Stages); t < issued; ++t)
            mbar_wait_bounded(is_k ? k8_full(t % kS8Div) : v8_full(t % kS8Div), (uint32_t)((t / kS8Div) & 1),
                              p.wait_limit_ns);
    } else if (!KV8 && warp >= 5 && n_tiles > 0) {
        // ---- copy warps: warp 5 streams K into its stages (lane 4x + h: 64-dim block h of box
        // x), warp 6 V (lane x: box x, all four blocks); the block-table entry of each box is read
        // a tile before its use
        const bool is_k = warp == 5;
        const int stages = is_k ? kKStages : kVStages;
        const uint64_t policy = l2_policy_evict_first();
        const int x = is_k ? lane >> 2 : lane, dc = is_k ? lane & 3 : 0;
        auto fetch = [&](int j) {
            const int key = (t0 + j) * KT + x * box_t;
            return (dc == 0 && x < nbox && j < n_tiles && key < n_keys)
                       ? p.block_table[(size_t)b * p.max_pages + (key >> p.log2P)]
                       : -1;
        };
        int raw = fetch(0);
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % stages;
            const int next_raw = fetch(j + 1);
            const bool has_key = x < nbox && (t0 + j) * KT + x * box_t < n_keys;
            const int pg_raw = is_k ? __shfl_sync(0xffffffffu, raw, lane & ~3) : raw;
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
                if (dc == 0 && x < nbox) sm_pg[(j % kTcPageRing) * 16 + x] = pg;
                __syncwarp();
            }
            const uint32_t full = is_k ? k_full(st) : v_full(st);
            const uint32_t copy_bytes = (uint32_t)box_t * (is_k ? 128u : 512u);
            if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)__popc(ok) * copy_bytes);
            __syncwarp();
            if (pg >= 0) {
                const int row = pg * p.P + (((t0 + j) * KT + x * box_t) & (p.P - 1));
                if (is_k)
                    tma_load_3d(sK(st) + (uint32_t)(dc * kKBlk + x * box_t * 128), &tmK, dc * 64, kvh, row, full,
                                policy);
                else
                    tma_load_4d(sV(st) + (uint32_t)(x * box_t * 512), &tmV, 0, row, 0, kvh, full, policy);
            }
            issued = j + 1;
            raw = next_raw;
        }
        // the last copies have landed before the CTA exits (consumed, or waited for here)
        for (int t = max(0, issued - stages); t < issued; ++t)
            mbar_wait_bounded(is_k ? k_full(t % stages) : v_full(t % stages), (uint32_t)((t / stages) & 1),
                              p.wait_limit_ns);
    } else if (warp == 4 && n_tiles > 0) {
        // ---- MMA warp: every lane waits, lane 0 issues
        const bool leader = lane == 0;
        // zeroes the V rows of tile j whose keys are invalid (past n_keys, bad page): key k is
        // row k % box_t of box k / box_t; lane = 8 h + c clears chunk c of 64-dim block h
        auto zero_invalid_v = [&](int j) {
            const int *ids = sm_pg + (j % kTcPageRing) * 16;
            const int first_past = min(KT, max(0, n_keys - (t0 + j) * KT));  // keys past n_keys: [first_past, KT)
            bool bad = false;  // a missing page among the keys before that
            for (int bx = 0; bx < nbox; ++bx) bad |= ids[bx] < 0 && (bx << log2box) < first_past;
            if (first_past == KT && !bad) return;
            const uint32_t dst = sV(j % kVStages) + (uint32_t)((lane >> 3) * box_t * 128 + (lane & 7) * 16);
            auto zero_key = [&](int k) {
                st_shared_v4(dst + (uint32_t)((k >> log2box) * box_t * 512 + (k & (box_t - 1)) * 128), 0u, 0u, 0u, 0u);
            };
            for (int k = first_past; k < KT; ++k) zero_key(k);
            if (bad)
                for (int bx = 0; bx < nbox; ++bx)
                    if (ids[bx] < 0 && (bx << log2box) < first_past)
                        for (int k = bx << log2box; k < min((bx + 1) << log2box, first_past); ++k) zero_key(k);
            fence_proxy_async_shared();
            __syncwarp();
        };
        // V operand of the 16-key MMA step kk (MN-major, N = 256 dims in four 64-dim blocks
        // box_t * 128 bytes apart): 8-key groups 1024 bytes apart within a box, or, with 8-key
        // boxes, one box (4096 bytes) per group
        auto v_desc = [&](uint32_t stage, int kk) {
            const int k0 = kk * 16;
            return box_t == 8 ? tc_desc(stage + (uint32_t)(kk * 8192), 1024, 4096)
                              : tc_desc(stage + (uint32_t)((k0 >> log2box) * box_t * 512 + (k0 & (box_t - 1)) * 128),
                                        (uint32_t)(box_t * 128), 1024);
        };
        constexpr uint32_t kIdS = tc_idesc_bf16(kTcRows, KT, false);
        constexpr uint32_t kIdO = tc_idesc_bf16(kTcRows, D, true);
        constexpr uint32_t kIdL = tc_idesc_bf16(kTcRows, 16, false);
        for (int j = 0; j <= n_tiles; ++j) {
            if (j < n_tiles) {  // S(j) = Q K(j)^T into S buffer j & 1
                const int ks = j % kKStages, sb = j & 1;
                if (!__all_sync(0xffffffffu,
                                (j > 0 || mbar_wait_bounded(q_full, 0, p.wait_limit_ns)) &&
                                    mbar_wait_bounded(k_full(ks), (uint32_t)((j / kKStages) & 1),
                                                      p.wait_limit_ns) &&
                                    (j < 2 || mbar_wait_bounded(s_free(sb), (uint32_t)(((j >> 1) - 1) & 1),
                                                                p.wait_limit_ns)))) {
                    failed = true;
                    break;
                }
                if (leader) {
                    tc_fence_after();
#pragma unroll
                    for (int dc = 0; dc < 4; ++dc)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_bf16(tS(sb), tc_desc(sQ + (uint32_t)(dc * kQBlk + k * 32), 16, 1024),
                                        tc_desc(sK(ks) + (uint32_t)(dc * kKBlk + k * 32), 16, 1024), kIdS,
                                        (dc | k) != 0);
                    tc_commit(s_full(sb));
                    tc_commit(k_empty(ks));
                    mbar_arrive(s_full(sb));
                }
                __syncwarp();
            }
            if (j >= 1) {  // O += P(j-1) V(j-1)
                const int t = j - 1, vs = t % kVStages;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(v_full(vs), (uint32_t)((t / kVStages) & 1),
                                                               p.wait_limit_ns))) {
                    failed = true;
                    break;
                }
                zero_invalid_v(t);
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(p_full, (uint32_t)(t & 1), p.wait_limit_ns))) {
                    failed = true;
                    break;
                }
                if (leader) {
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk) {
                        tc_mma_bf16_ts(tO, tP + (uint32_t)(kk * 8), v_desc(sV(vs), kk), kIdO, t > 0 || kk > 0);
                        tc_mma_bf16_ts(tL, tP + (uint32_t)(kk * 8), tc_desc(sOnes + (uint32_t)(kk * 32), 16, 1024),
                                       kIdL, t > 0 || kk > 0);
                    }
                    tc_commit(o_done);
                    tc_commit(v_empty(vs));
                }
                __syncwarp();
            }
        }
        // the MMAs in flight finish before the CTA exits
        if (leader) {
            tc_commit(drain);
            if (!mbar_wait_bounded(drain, 0, p.wait_limit_ns)) failed = true;
        }
    } else if (!issuer_warp && n_tiles > 0) {
        // ---- softmax warps: thread r owns row r.  Q rows (128B-swizzled [4 column blocks][128
        // rows][128 B]) and the ones tile into shared memory first, while the copies start.
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + grow * D);
#pragma unroll
            for (int cq = 0; cq < 32; ++cq) {
                const uint4 v = row_ok ? __ldg(src + cq) : make_uint4(0u, 0u, 0u, 0u);
                const int dc = cq >> 3, cc = cq & 7;
                st_shared_v4(sQ + (uint32_t)(dc * kQBlk + r * 128 + ((cc ^ (r & 7)) << 4)), v.x, v.y, v.z, v.w);
            }
            constexpr uint32_t kOne2 = 0x3F803F80u;  // two bf16 ones
            st_shared_v4(sOnes + (uint32_t)(r * 16), kOne2, kOne2, kOne2, kOne2);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        const float c = p.scale_log2;  // > 0
        float m_ref = kNegInf, l_run = 0.f;
        const int row_lim = min(n_keys, klim + 1);  // keys [0, row_lim) are visible to this row
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full(sb), (uint32_t)((j >> 1) & 1), p.wait_limit_ns))) {
                failed = true;
                break;
            }
            tc_fence_after();
            uint32_t sr[KT];
            tc_ld64(tS(sb) + lane_off, sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(sb));
            // masking: none on tiles every row of the warp sees whole, the row's limit on
            // the diagonal, a key bitmask where a page is missing
            const int *ids = sm_pg + (j % kTcPageRing) * 16;
            bool pages_ok = true;
            for (int x = 0; x < nbox; ++x) pages_ok &= ids[x] >= 0;
            const int lim = row_lim - (t0 + j) * KT;
            if (!pages_ok) {
                uint32_t okw0 = 0u, okw1 = 0u;
                for (int x = 0; x < nbox; ++x) {
                    if (ids[x] < 0) continue;
                    const int k0 = x << log2box, k1 = k0 + box_t;
                    for (int w = k0 >> 5; w < ((k1 + 31) >> 5); ++w) {
                        const int lo = max(k0, 32 * w) - 32 * w, n = min(k1, 32 * w + 32) - 32 * w - lo;
                        const uint32_t bits = (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) << lo;
                        if (w == 0) okw0 |= bits;
                        else okw1 |= bits;
                    }
                }
#pragma unroll
                for (int i = 0; i < KT; ++i)
                    if (!((((i < 32) ? okw0 : okw1) >> (i & 31)) & 1u) || i >= lim) sr[i] = 0xff800000u;  // -inf
            } else if (__any_sync(0xffffffffu, lim < KT)) {
#pragma unroll
                for (int i = 0; i < KT; ++i)
                    if (i >= lim) sr[i] = 0xff800000u;
            }
            // tile maximum of the unscaled scores, eight chains
            float mx8[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) mx8[a] = __uint_as_float(sr[a]);
#pragma unroll
            for (int i = 8; i < KT; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
            const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                             c;
            // reference maximum: set at the first visible key, moved only past a 2^8 rise
            float alpha = 1.f;
            if (mx != kNegInf && (m_ref == kNegInf || mx > m_ref + kRescaleGap)) {
                alpha = m_ref == kNegInf ? 0.f : ex2(m_ref - mx);
                m_ref = mx;
                l_run *= alpha;
            }
            const float neg_ref = m_ref == kNegInf ? 0.f : -m_ref;
            float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pw[KT / 2];
#pragma unroll
            for (int i = 0; i < KT / 2; ++i) {
                const float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), c, neg_ref));
                const float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), c, neg_ref));
                pw[i] = pack_bf16x2(p0, p1);
                ls[i & 7] += p0 + p1;
            }
            l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
            // PV(j-1) must be done before O is rescaled and the P buffer rewritten
            if (j >= 1) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done, (uint32_t)((j - 1) & 1), p.wait_limit_ns))) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int cb = 0; cb < D / 32; ++cb) {
                        float v[32];
                        tc_ld32(tO + lane_off + (uint32_t)(cb * 32), v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= alpha;
                        tc_st32(tO + lane_off + (uint32_t)(cb * 32), v);
                    }
                    tc_st1(tL + lane_off, tc_ld1(tL + lane_off) * alpha);
                }
            }
            // P (bf16 pairs) into this row's lane of tensor memory
            tc_st32u(tP + lane_off, pw);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        // epilogue: out = O / lt, lse = (m + log2 l) ln 2
        if (!failed &&
            !__all_sync(0xffffffffu, mbar_wait_bounded(o_done, (uint32_t)((n_tiles - 1) & 1), p.wait_limit_ns)))
            failed = true;
        if (!failed) {
            tc_fence_after();
            const bool empty = m_ref == kNegInf;
            const float lt = tc_ld1(tL + lane_off);  // collective: every lane loads
            const float inv = empty ? 0.f : 1.f / lt;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + grow * D);
            const float row_lse = empty ? kNegInf : (m_ref + __log2f(l_run)) * 0.693147180559945309f;
#pragma unroll
            for (int cb = 0; cb < D / 32; ++cb) {
                float v[32];
                tc_ld32(tO + lane_off + (uint32_t)(cb * 32), v);
                if (row_ok && direct) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[cb * 4 + i] = make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                                     pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                                     pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                                     pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
                } else if (row_ok) {
                    t256_store_partial(p, split, grow, cb, v, inv);
                }
            }
            if (row_ok && direct && p.lse) p.lse[grow] = row_lse;
            if (row_ok && !direct) p.part_lse[split * p.total_rows + grow] = row_lse;
        }
    }
    if (!issuer_warp && n_tiles == 0 && row_ok) {  // no key visible to the CTA: out = 0, lse = -inf
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
        int *last = reinterpret_cast<int *>(smem_raw + Smem::tmem_slot + 4);
        __threadfence();
        __syncthreads();
        if (tid == 0)
            *last = atomicInc(reinterpret_cast<unsigned *>(p.counters + ((size_t)b * p.q_tiles + qt) * p.Hkv + kvh),
                              (unsigned)(n_chunks - 1)) == (unsigned)(n_chunks - 1);
        __syncthreads();
        if (*last) {  // every warp merges rows warp, warp + W, ... of this CTA
            __threadfence();
            for (int cr = warp; cr < nrows; cr += kThreads / 32) {
                const int rt = (row0 + cr) / G, rh = (row0 + cr) % G;
                t256_merge_row_warp(p, n_chunks, (size_t)(q_base + rt) * p.Hq + kvh * G + rh, lane);
            }
        }
    }
}

}  // namespace pkv
