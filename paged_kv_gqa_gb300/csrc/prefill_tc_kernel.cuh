// prefill_tc_kernel.cuh -- several query rows per sequence on the 5th-generation tensor
// cores (tcgen05), for groups of more than 32 rows (chunked prefill, multi-token steps over
// long tables); a bf16 cache, or an fp8 (e4m3) one (the KV8 instantiation: see TcCfg).
//
// One CTA per 128 (token, query head) rows of one (sequence, kv head) group, the rows
// packed token-major as in the multi-row decode kernel (AstrAI "CUDA Kernels", "Q
// Scheduling and KV Addressing": the query heads of one kv-head group share each K/V
// tile).  The CTA walks the keys its rows may see in tiles of 128:
//     S  = Q K^T       tcgen05.mma M=128 rows, N=128 keys, K=D; S in tensor memory
//     softmax          thread r of the softmax warps owns row r = TMEM lane r: the row
//                      maximum and sums need no shuffles
//     O += P V         tcgen05.mma M=128 rows, N=D, K=128 keys; O in tensor memory
// Warp specialisation: warps 0-3 run the softmax, one lane of warp 4 issues the MMAs,
// warp 5 copies K and warp 6 copies V (TMA; every lane issues one 16-key box half, as
// one thread's copies issue too slowly to feed the tensor cores from page-sized boxes).
// S is double-buffered in tensor memory, so the score MMA of tile j+1 runs while the
// softmax warps work on tile j, and the PV MMA of tile j runs while they load and
// exponentiate tile j+1.  K and V have three shared-memory stages each (bf16 cache; the
// fp8 instantiation's stages are in TcCfg).  mbarriers hand
// every buffer over (copies: complete_tx; MMAs: tcgen05.commit; softmax: one arrival
// per warp).
// The online softmax keeps a reference maximum per row and moves it only when a tile's
// maximum exceeds it by more than 2^8 (probabilities stay <= 256, well inside f32 and
// bf16), so O is rescaled in tensor memory (tcgen05.ld/st) only then; l and O share the
// reference, so the result is the same softmax.  The sum of the bf16-rounded
// probabilities that normalises O comes from the tensor cores too: one more MMA per key
// tile multiplies P by a column of ones into a 16-column accumulator beside O.  The f32
// sum l, kept by the softmax threads, gives the log-sum-exp.  The scores' scale must be
// positive (the host routes other scales elsewhere): the row maximum is then taken on
// the unscaled scores and each exponent is one FMA.
// Q and K tiles sit in shared memory 128B-swizzled, K-major ([D/64][rows][64]) as the
// TMA boxes land them (two copies, one per 64 dims, per page box).  V is read MN-major
// (N = dims contiguous) in the layout one copy per page box lands: [box][D/64][keys][64].
// P (bf16) goes from the softmax threads' registers to tensor memory (tcgen05.st) and
// is the A operand of the PV MMA there.  Keys past the last one the CTA's rows may see, or
// in a page whose id is out of range, are masked in the scores and zeroed in V's rows
// by the issuing lane before the PV MMA (0 * NaN would reach the output).  Every wait is
// bounded; on a timeout the status word is set, the issuing lane waits (bounded) for its
// copies and MMAs in flight, and every warp stops.
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
    // key splits: a CTA takes chunk_tiles key tiles of its group; a group with more than
    // one chunk writes per-split partials and its last split merges them
    float *part_lse;         // [splits, total_q * Hq] natural-log lse of each split
    float *part_out;         // [splits, total_q * Hq, D] each split's normalised output
    int *counters;           // [B, q_tiles, Hkv] splits finished per group (wraps to 0 after the last)
    size_t total_rows;       // total_q * Hq
    // fp8 (e4m3) cache: per-(page, kv head, slot) power-of-two scales [num_pages, Hkv, P]
    // (the codes' pools come through the tensor maps); unused with a bf16 cache
    const float *k_scale, *v_scale;
    int chunk_tiles;
    int B, Hq, Hkv, G, P, log2P, num_pages, max_pages, total_q, max_q_len, causal, q_tiles;
    float scale_log2;
    unsigned long long wait_limit_ns;
};

// The last split of a group to finish merges the splits' partial outputs of one row with the
// log-sum-exp recurrence (FlashQuant wiki "CUDA Kernels", split_k_reduce.cu "Algorithm":
// split s weighs exp(lse_s - max lse)), in split order.  One warp per row: lane l owns dims
// 4l .. 4l + 3, so each split's partial row is one coalesced 512-byte load; lane s % 32
// computes split s's weight, eight splits' loads are in flight at a time.
__device__ __forceinline__ void tc_merge_row_warp(const PrefillTcParams &p, int n_chunks, size_t grow, int lane)
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
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n_chunks; c0 += 32) {
        // weight of split c0 + lane, broadcast below
        const float wl = c0 + lane < n_chunks
                             ? ex2((__ldcg(p.part_lse + (c0 + lane) * p.total_rows + grow) - mr) * kLog2e) * inv
                             : 0.f;
        const int nc = min(32, n_chunks - c0);
        for (int k0 = 0; k0 < nc; k0 += 8) {
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                v[k] = k0 + k < nc ? __ldcg(reinterpret_cast<const float4 *>(
                                              p.part_out + ((size_t)(c0 + k0 + k) * p.total_rows + grow) * 128) +
                                          lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, (k0 + k) & 31);
                a.x += v[k].x * w;
                a.y += v[k].y * w;
                a.z += v[k].z * w;
                a.w += v[k].w * w;
            }
        }
    }
    reinterpret_cast<uint2 *>(p.out + grow * 128)[lane] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    if (lane == 0 && p.lse) p.lse[grow] = m == ninf ? ninf : m + __logf(wsum);
}

// A split's row result into the partials (O / lt in f32, natural-log lse); o holds 32 of
// the row's 128 dims, columns 32 cb .. 32 cb + 31.
__device__ __forceinline__ void tc_store_partial(const PrefillTcParams &p, int c, size_t grow, int cb,
                                                 const float (&o)[32], float inv)
{
    float4 *dst = reinterpret_cast<float4 *>(p.part_out + (c * p.total_rows + grow) * 128) + cb * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
}

constexpr int kTcRows = 128;     // rows per CTA (the MMA's M)
constexpr int kTcKeys = 128;     // keys per tile (the score MMA's N)
constexpr int kTcPageRing = 8;   // tiles whose page ids are kept

// Per cache type: threads, bf16 K and V stages, fp8 staging stages.  bf16: 4 softmax warps,
// the MMA warp, the K and V copy warps; K and V land by TMA straight into three stages each.
// fp8: the copy warps land the e4m3 codes and scales in two staging stages, and two K and two
// V converter warps (7-8, 9-10) write them, dequantised to bf16, into the layout the bf16
// copies land: one K stage (a key tile's K is written once the previous tile's score MMA has
// read the stage, which it does about a tile ahead of the softmax) and two V stages (V waits on
// the PV products, issued only after the softmax); measured on GB300 9-12% faster than two K
// stages and one V stage.
template <bool KV8>
struct TcCfg {
    static constexpr int threads = KV8 ? 352 : 224;
    static constexpr int k_stages = KV8 ? 1 : 3;
    static constexpr int v_stages = KV8 ? 2 : 3;
    static constexpr int s8_stages = KV8 ? 2 : 0;
};
constexpr int kTcThreads = TcCfg<false>::threads;
constexpr int kTc8Threads = TcCfg<true>::threads;

// Shared memory (bytes from a 1024-aligned base) of the D = 128 kernel.
template <bool KV8>
struct TcSmemT {
    static constexpr int kTile = kTcRows * 128 * 2;  // 128 rows x 128 dims (or keys) bf16, 2 column blocks
    static constexpr int kCodes = kTcKeys * 128;      // 128 keys x 128 e4m3 codes
    // fp8 staging stage: [K codes][V codes] (each as the 128B-swizzled page boxes land) [K scales][V scales]
    static constexpr int kStage8 = 2 * kCodes + 2 * kTcKeys * 4;
    static constexpr int q = 0;
    static constexpr int k = kTile;                                      // K stage s at k + s * kTile
    static constexpr int v = k + TcCfg<KV8>::k_stages * kTile;           // V stage s at v + s * kTile
    static constexpr int ones = v + TcCfg<KV8>::v_stages * kTile;        // 16 x 64 bf16 ones, the B operand of the row-sum MMA
    static constexpr int s8 = (ones + 2048 + 1023) / 1024 * 1024;       // fp8 staging stage s at s8 + s * kStage8
    static constexpr int bars = s8 + TcCfg<KV8>::s8_stages * kStage8;    // 32 mbarriers
    static constexpr int pages = bars + 32 * 8;                          // [kTcPageRing][16] page id of each box, -1: none
    static constexpr int tmem_slot = pages + kTcPageRing * 16 * 4;
    static constexpr int total = tmem_slot + 16;
    static constexpr int dynamic = total;                                // the dynamic shared memory starts 1024-aligned
};
using TcSmem = TcSmemT<false>;
using Tc8Smem = TcSmemT<true>;
static_assert(TcSmem::dynamic <= 232448 && Tc8Smem::dynamic <= 232448,
              "prefill_tc_kernel: shared memory above the per-block limit");
static_assert(Tc8Smem::kStage8 % 1024 == 0, "prefill_tc_kernel: fp8 staging stages must stay 1024-aligned");

// 16 bytes of shared memory, kept in order with the mbarrier waits around it.
__device__ __forceinline__ uint4 tc_ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// 16 e4m3 codes (byte 0 first) times a power-of-two scale -> 16 bf16 in 8 pairs (element 2i
// in the low half of o[i]): e4m3 -> f16 and f16 -> f32 are exact, the product is exact
// while it stays a normal f32, and its rounding to bf16 is the one a bf16 copy of the
// dequantised cache holds.
__device__ __forceinline__ void e4m3x16_scaled_to_bf16(const uint4 c, float s, uint32_t (&o)[8])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h01, h23;
        e4m3x4_to_f16x2x2(w[i], h01, h23);
        float a0, a1, a2, a3;
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
            : "=f"(a0), "=f"(a1)
            : "r"(h01));
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
            : "=f"(a2), "=f"(a3)
            : "r"(h23));
        o[2 * i] = pack_bf16x2(a0 * s, a1 * s);
        o[2 * i + 1] = pack_bf16x2(a2 * s, a3 * s);
    }
}

template <bool KV8>
__global__ void __launch_bounds__(TcCfg<KV8>::threads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const PrefillTcParams p)
{
    constexpr int D = 128;
    using Smem = TcSmemT<KV8>;
    constexpr int kThreads = TcCfg<KV8>::threads;
    constexpr int kTcKStages = TcCfg<KV8>::k_stages;
    constexpr int kTcVStages = TcCfg<KV8>::v_stages;
    constexpr int kS8Stages = TcCfg<KV8>::s8_stages;
    constexpr int kS8Div = kS8Stages > 0 ? kS8Stages : 1;  // the bf16 instantiation compiles the fp8 roles too
    constexpr int kTile = Smem::kTile;
    constexpr int kBlk = kTcRows * 128;  // bytes of one 64-column block of a tile
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
    uint8_t *sbase = smem_raw;
    const uint32_t sQ = base + Smem::q, sOnes = base + Smem::ones;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + Smem::bars);
    int *sm_pg = reinterpret_cast<int *>(sbase + Smem::pages);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sbase + Smem::tmem_slot);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    constexpr int kKFull = 0, kKEmpty = kKFull + kTcKStages, kVFull = kKEmpty + kTcKStages,
                  kVEmpty = kVFull + kTcVStages, kSFull = kVEmpty + kTcVStages, kSFree = kSFull + 2,
                  kPFull = kSFree + 2, kODone = kPFull + 1, kDrain = kODone + 1, kQFull = kDrain + 1,
                  kK8Full = kQFull + 1, kK8Empty = kK8Full + kS8Stages, kV8Full = kK8Empty + kS8Stages,
                  kV8Empty = kV8Full + kS8Stages, kBarEnd = kV8Empty + kS8Stages;
    static_assert(kBarEnd <= 32, "prefill_tc_kernel: more mbarriers than the shared-memory slots");
    auto k_full = [&](int s) { return bar(kKFull + s); };
    auto k_empty = [&](int s) { return bar(kKEmpty + s); };
    auto v_full = [&](int s) { return bar(kVFull + s); };
    auto v_empty = [&](int s) { return bar(kVEmpty + s); };
    auto s_full = [&](int s) { return bar(kSFull + s); };
    auto s_free = [&](int s) { return bar(kSFree + s); };
    const uint32_t p_full = bar(kPFull), o_done = bar(kODone), drain = bar(kDrain), q_full = bar(kQFull);
    auto k8_full = [&](int s) { return bar(kK8Full + s); };     // fp8: codes and scales of a staging stage landed
    auto k8_empty = [&](int s) { return bar(kK8Empty + s); };   // fp8: the converters have read the stage
    auto v8_full = [&](int s) { return bar(kV8Full + s); };
    auto v8_empty = [&](int s) { return bar(kV8Empty + s); };
    auto sK = [&](int s) { return base + Smem::k + (uint32_t)(s * kTile); };
    auto sV = [&](int s) { return base + Smem::v + (uint32_t)(s * kTile); };
    auto s8 = [&](int s) { return base + Smem::s8 + (uint32_t)(s * Smem::kStage8); };

    if (tid == 0) {
        // bf16: a full K/V stage is the copy lane's expect_tx; fp8: one arrival per converter warp
        for (int s = 0; s < kTcKStages; ++s) {
            mbar_init(k_full(s), KV8 ? 2 : 1);
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < kTcVStages; ++s) {
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
    // TMEM columns: S0 0..127, S1 128..255, O 256..383, the row sums of bf16 P 384..399,
    // P (bf16 pairs) 448..511
    if (warp == 0) tc_alloc(smem_addr(tmem_slot), 512);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + 256u, tL = tmem + 384u, tP = tmem + 448u;
    auto tS = [&](int sb) { return tmem + (uint32_t)(sb * 128); };
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int log2box = p.log2P < 7 ? p.log2P : 7;
    const int box_t = 1 << log2box;
    const int nbox = kTcKeys / box_t;
    bool failed = false;

    if (KV8 && warp >= 7 && n_tiles > 0) {
        // ---- fp8 converter warps: 7-8 write K tiles, 9-10 V tiles.  A task is 16 codes (one
        // 16-byte chunk of a key row): read unswizzled from the staging box, scaled to bf16, and
        // stored as the two 16-byte chunks the bf16 copies would land (128B swizzle on the
        // row's address bits 7-9)
        const bool is_k = warp < 9;
        const int ct = (warp - (is_k ? 7 : 9)) * 32 + lane;  // 0..63
        for (int j = 0; j < n_tiles; ++j) {
            const int st8 = j % kS8Div;
            const bool ok = mbar_wait_bounded(is_k ? k8_full(st8) : v8_full(st8), (uint32_t)((j / kS8Div) & 1),
                                              p.wait_limit_ns) &&
                            (is_k ? (j < kTcKStages || mbar_wait_bounded(k_empty(j % kTcKStages),
                                                                          (uint32_t)((j / kTcKStages - 1) & 1),
                                                                          p.wait_limit_ns))
                                  : (j < kTcVStages || mbar_wait_bounded(v_empty(j % kTcVStages),
                                                                          (uint32_t)((j / kTcVStages - 1) & 1),
                                                                          p.wait_limit_ns)));
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                break;
            }
            const uint32_t src = s8(st8) + (is_k ? 0u : (uint32_t)Smem::kCodes);
            const uint32_t scl = s8(st8) + (uint32_t)(2 * Smem::kCodes) + (is_k ? 0u : (uint32_t)(kTcKeys * 4));
            const uint32_t dst = is_k ? sK(j % kTcKStages) : sV(j % kTcVStages);
#pragma unroll 4
            for (int t = ct; t < kTcKeys * 8; t += 64) {
                const int key = t >> 3, ch = t & 7, sw = key & 7;
                const uint4 c = tc_ld_shared_v4(src + (uint32_t)(key * 128 + ((ch ^ sw) << 4)));
                uint32_t o[8];
                e4m3x16_scaled_to_bf16(c, ld_shared_f32(scl + (uint32_t)(key * 4)), o);
                // K: [64-dim block][key][128 B]; V: [box][64-dim block][key in box][128 B]
                const int half = ch >> 2, c16 = (ch & 3) * 2;
                const uint32_t row = is_k ? dst + (uint32_t)(half * kBlk + key * 128)
                                          : dst + (uint32_t)((key >> log2box) * box_t * 256 + half * box_t * 128 +
                                                             (key & (box_t - 1)) * 128);
                st_shared_v4(row + (uint32_t)((c16 ^ sw) << 4), o[0], o[1], o[2], o[3]);
                st_shared_v4(row + (uint32_t)(((c16 + 1) ^ sw) << 4), o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_shared();  // the MMAs read the tile through the async proxy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(is_k ? k_full(j % kTcKStages) : v_full(j % kTcVStages));
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
            const int key = (t0 + j) * kTcKeys + x * box_t;
            return (x < nbox && j < n_tiles && key < n_keys) ? p.block_table[(size_t)b * p.max_pages + (key >> p.log2P)]
                                                            : -1;
        };
        int raw = fetch(0);
        int issued = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j % kS8Div;
            const int next_raw = fetch(j + 1);
            const bool has_key = x < nbox && (t0 + j) * kTcKeys + x * box_t < n_keys;
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
            if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)__popc(ok) * (uint32_t)box_t * (128u + 4u));
            __syncwarp();
            if (pg >= 0) {
                const int slot = ((t0 + j) * kTcKeys + x * box_t) & (p.P - 1);
                const uint32_t codes = s8(st) + (is_k ? 0u : (uint32_t)Smem::kCodes) + (uint32_t)(x * box_t * 128);
                tma_load_4d(codes, is_k ? &tmK : &tmV, 0, pg * p.P + slot, 0, kvh, full, policy);
                const uint32_t sdst = s8(st) + (uint32_t)(2 * Smem::kCodes) + (is_k ? 0u : (uint32_t)(kTcKeys * 4)) +
                                      (uint32_t)(x * box_t * 4);
                bulk_copy_g2s(sdst, (is_k ? p.k_scale : p.v_scale) + ((size_t)pg * p.Hkv + kvh) * p.P + slot,
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
        // ---- copy warps: warp 5 streams K into its 3 stages, warp 6 V into its 3; lane
        // 2x + h copies half h (64 dims) of box x (box_t keys of one page)
        const bool is_k = warp == 5;
        const int stages = is_k ? kTcKStages : kTcVStages;
        const uint64_t policy = l2_policy_evict_first();
        // K: lane 2x + h copies half h (64 dims) of box x; V: lane x copies box x whole
        const int x = is_k ? lane >> 1 : lane, dc = is_k ? lane & 1 : 0;
        // block-table entry of box x of tile j (lanes x < nbox), read a tile before its use
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
                if (dc == 0 && x < nbox) sm_pg[(j % kTcPageRing) * 16 + x] = pg;
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
    } else if (warp == 4 && n_tiles > 0) {
        // ---- MMA warp: every lane waits, lane 0 issues
        const bool leader = lane == 0;
        // zeroes the V rows of tile j whose keys are invalid (past n_keys, bad page): key k
        // is row k % box_t of box k / box_t, 2 halves x 8 chunks of 16 bytes; lanes 0-15
        // clear the even keys, 16-31 the odd ones, lane & 15 naming the chunk
        auto zero_invalid_v = [&](int j) {
            const int *ids = sm_pg + (j % kTcPageRing) * 16;
            const int first_past = min(kTcKeys, max(0, n_keys - (t0 + j) * kTcKeys));  // keys past n_keys: [first_past, 128)
            bool bad = false;  // a missing page among the keys before that
            for (int bx = 0; bx < nbox; ++bx) bad |= ids[bx] < 0 && (bx << log2box) < first_past;
            if (first_past == kTcKeys && !bad) return;
            const uint32_t dst = sV(j % kTcVStages) + (uint32_t)(((lane >> 3) & 1) * box_t * 128 + (lane & 7) * 16);
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
        constexpr uint32_t kIdS = tc_idesc_bf16(kTcRows, kTcKeys, false);
        constexpr uint32_t kIdO = tc_idesc_bf16(kTcRows, D, true);
        constexpr uint32_t kIdL = tc_idesc_bf16(kTcRows, 16, false);
        for (int j = 0; j <= n_tiles; ++j) {
            if (j < n_tiles) {  // S(j) = Q K(j)^T into S buffer j & 1
                const int ks = j % kTcKStages, sb = j & 1;
                if (!__all_sync(0xffffffffu,
                                (j > 0 || mbar_wait_bounded(q_full, 0, p.wait_limit_ns)) &&
                                    mbar_wait_bounded(k_full(ks), (uint32_t)((j / kTcKStages) & 1), p.wait_limit_ns) &&
                                    (j < 2 || mbar_wait_bounded(s_free(sb), (uint32_t)(((j >> 1) - 1) & 1),
                                                                p.wait_limit_ns)))) {
                    failed = true;
                    break;
                }
                if (leader) {
                    tc_fence_after();
#pragma unroll
                    for (int dc = 0; dc < 2; ++dc)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_bf16(tS(sb), tc_desc(sQ + (uint32_t)(dc * kBlk + k * 32), 16, 1024),
                                        tc_desc(sK(ks) + (uint32_t)(dc * kBlk + k * 32), 16, 1024), kIdS,
                                        (dc | k) != 0);
                    tc_commit(s_full(sb));
                    tc_commit(k_empty(ks));
                    mbar_arrive(s_full(sb));
                }
                __syncwarp();
            }
            if (j >= 1) {  // O += P(j-1) V(j-1)
                const int t = j - 1, vs = t % kTcVStages;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(v_full(vs), (uint32_t)((t / kTcVStages) & 1),
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
                    for (int kk = 0; kk < 8; ++kk) {
                        tc_mma_bf16_ts(tO, tP + (uint32_t)(kk * 8), v_desc(sV(vs), kk), kIdO, t > 0 || kk > 0);
                        tc_mma_bf16_ts(tL, tP + (uint32_t)(kk * 8), tc_desc(sOnes + (uint32_t)((kk & 3) * 32), 16, 1024),
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
    } else if (n_tiles > 0) {
        // ---- softmax warps: thread r owns row r.  Q rows (128B-swizzled [2 column blocks][128
        // rows][128 B]) and the ones tile into shared memory first, while the copies start.
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + grow * D);
#pragma unroll
            for (int cq = 0; cq < 16; ++cq) {
                const uint4 v = row_ok ? __ldg(src + cq) : make_uint4(0u, 0u, 0u, 0u);
                const int dc = cq >> 3, cc = cq & 7;
                st_shared_v4(sQ + (uint32_t)(dc * kBlk + r * 128 + ((cc ^ (r & 7)) << 4)), v.x, v.y, v.z, v.w);
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
            uint32_t sr[kTcKeys];
            tc_ld128(tS(sb) + lane_off, sr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(sb));
            // masking: none on tiles every row of the warp sees whole, the row's limit on
            // the diagonal, a key bitmask where a page is missing
            const int *ids = sm_pg + (j % kTcPageRing) * 16;
            bool pages_ok = true;
            for (int x = 0; x < nbox; ++x) pages_ok &= ids[x] >= 0;
            const int lim = row_lim - (t0 + j) * kTcKeys;
            if (!pages_ok) {
                uint32_t okw[4] = {0u, 0u, 0u, 0u};
                for (int x = 0; x < nbox; ++x) {
                    if (ids[x] < 0) continue;
                    const int k0 = x << log2box, k1 = k0 + box_t;
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
            // tile maximum of the unscaled scores, eight chains
            float mx8[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) mx8[a] = __uint_as_float(sr[a]);
#pragma unroll
            for (int i = 8; i < kTcKeys; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(sr[i]));
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
            uint32_t pw[kTcKeys / 2];
#pragma unroll
            for (int i = 0; i < kTcKeys / 2; ++i) {
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
                    for (int cb = 0; cb < 4; ++cb) {
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
            tc_st64(tP + lane_off, pw);
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
            for (int cb = 0; cb < 4; ++cb) {
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
                    tc_store_partial(p, split, grow, cb, v, inv);
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
        int *last = reinterpret_cast<int *>(sbase + Smem::tmem_slot + 4);
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
                tc_merge_row_warp(p, n_chunks, (size_t)(q_base + rt) * p.Hq + kvh * G + rh, lane);
            }
        }
    }
}

}  // namespace pkv
