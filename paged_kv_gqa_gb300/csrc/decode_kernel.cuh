// decode_kernel.cuh -- split-KV paged GQA decode kernel for sm_103a.
//
// One thread block per (kv head, split c, sequence b).  The block owns the keys
// [c*chunk, min((c+1)*chunk, L_b)) of that kv head and all G = Hq/Hkv query
// heads that read it, so every K/V byte is fetched from HBM once per call
// (AstrAI "CUDA Kernels", "Q Scheduling and KV Addressing": packing the query
// heads of one kv-head group into a block streams K/V once per block rather
// than once per query head).
//
// Data movement.  Each of the W warps streams its own sequence of stages
// (stage s of the block goes to warp s % W).  A stage is T consecutive keys of
// one kv head, fetched by TMA straight out of the page pool: a rank-4 tensor
// map views k_cache/v_cache as (64 dims, num_pages*P rows, D/64 column blocks,
// Hkv heads), and one box (64, min(T,P), D/64, 1) moves a whole page slice of
// one head -- one copy per tensor per stage, with no per-thread address
// arithmetic.  (A rank-3 view with one box per 64 columns is the fallback.)  The physical row of a
// key is block_table[b][j >> log2 P] * P + (j & (P-1)) (FlashQuant wiki "CUDA
// Kernels", paged_decode.cu "Page Table Addressing": shift and mask instead of
// divide and modulo).  The block's slice of the block table is staged in shared
// memory first, so the page-id lookup is not a dependent global load in front
// of every copy.  Each warp keeps R stages in flight on its own mbarriers; lane
// 0 refills a slot as soon as the warp has consumed it.  Boxes land 128B-
// swizzled so the ldmatrix reads below are free of bank conflicts.
//
// Math.  Keys sit on the mma M dimension and the query heads of the group on N
// (8 per tile, padded), so G = 4, 8, 16 map onto m16n8k16 tiles without
// wasting rows:
//     S^T[key, head]  = K[key, :] . q^T[:, head]            (K via ldmatrix, q in registers)
//     O^T[d, head]   += V^T[d, key] . P^T[key, head]        (V via ldmatrix.trans)
// P^T comes out of the S accumulators as bf16 pairs and is turned into the B
// operand with movmatrix.trans.  The softmax is the online recurrence in base 2
// (FlashQuant wiki "CUDA Kernels", flash_attention.cu "Online Softmax"; the
// "exp2/log2(e) prescaling" row of its optimisation summary): scores are
// multiplied by scale*log2(e) in f32, the running max m, denominator l and the
// accumulators are f32, and every exponential is one ex2.approx.  Row maxima
// use warp shuffles; the denominators are summed per thread and reduced once at
// the end.  Two denominators are kept: the sum of the f32 probabilities, which
// gives the LSE, and the sum of the same bf16-rounded probabilities that feed
// the PV product, which normalises the output so that it is a convex
// combination of V rows up to f32 rounding (a constant V comes back unchanged).
//
// Masking.  Keys at or past L_b (the padded tail of the last page) and keys of
// a page whose id is out of range get score -inf, and their V values are
// zeroed in registers before the PV mma, so NaN or Inf left in unused slots
// never reaches the result (0 * NaN would).
//
// FP8 cache (KV8).  The pool may instead hold float8 e4m3 codes with one f32
// scale per (token, kv head), the scales stored [page][kv head][slot] so that a
// page slice of one head's scales is contiguous (OASR "Kernel Layer", "FP8 KV
// variants").  The ring carries the code bytes (one TMA box per tensor, 128B-
// swizzled like the bf16 tiles; 64B for D = 64) and the scales (one bulk copy per
// tensor) on the same mbarrier.  The codes go straight from shared memory into the
// mma fragments: ldmatrix on the code bytes (a b16 view: four codes per lane per
// 8x8 matrix), one cvt.rn.f16x2.e4m3x2 per code pair (exact: every e4m3 value is an
// f16), and the f16 mma.  No dequantised copy is written back to shared memory.
//   - Scores: a lane's four codes from one 16-byte chunk are its k slots
//     {2t, 2t+1, 2t+8, 2t+9}, so the query columns are permuted the same way within
//     each 16-wide k step (the same products, in other k slots).  q is held as f16
//     scaled by 2^eq, eq chosen per block so the group's largest |q| lands in
//     [2^14, 2^15) (exact for every element within 2^28 of it); the per-key K
//     scale and 2^-eq fold into the factor that turns scores into log2 units.
//   - Values: ldmatrix.trans on the code bytes gives a lane two keys x two
//     adjacent dims; one byte permute makes key pairs per dim, so the PV tile's
//     rows {g, g+8} are dims {2g, 2g+1} of each 16-dim chunk (only the output
//     rows' order changes).  The per-key V scale folds into the probabilities:
//     p * vscale * 2^-Ev, with Ev the running maximum of the scale exponents; a
//     rise of Ev rescales the accumulators along with the softmax correction, and
//     the warp's result is multiplied by 2^Ev at the end.  The f32 denominator
//     normalises the output.
// The pages' own design dequantises each stage into a served-dtype tile in shared
// memory; on this part that round trip through shared memory made the fp8 kernel
// slower than the bf16 one, so the fp8 path reads the codes in place instead.
//
// Epilogue.  The W warps' states are merged through shared memory.  If the
// sequence has a single split the block writes bf16 out and the natural-log
// lse directly; otherwise it writes its normalised f32 output and lse to the
// workspace (FlashQuant wiki "CUDA Kernels", paged_decode.cu "Partial Output";
// here normalised and in natural log), and the last split of the (b, kv head)
// group to finish merges the group's partials in the same launch, so no second
// kernel and no launch gap sit on the critical path; on a grid of one wave with
// 2-8 splits the splits of a group form a thread-block cluster instead and send
// their partials into split 0's shared memory, which merges them the same way.
// A split that starts past L_b exits at once and is never merged ("Early Exit for
// Empty Splits").  A decode group wider than one block (G = 32 at D = 256) runs on
// the several-rows instantiation with one row per sequence (no qo_indptr).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "plan.h"
#include "ptx.cuh"

namespace pkv {

struct DecodeParams {
    const __nv_bfloat16 *q;  // [B, Hq, D]
    const int *block_table;  // [B, max_pages]
    const int *seq_lens;     // [B]
    __nv_bfloat16 *out;      // [B, Hq, D]
    float *lse;              // [B, Hq] or nullptr
    float *part_lse;         // [S, B, Hq]
    float *part_out;         // [S, B, Hq, D]
    int *counters;           // [B, Hkv] splits finished per group (wraps to 0 after the last)
    int *status;             // workspace status word
    const float *k_scale;    // fp8 cache: [num_pages, Hkv, P] f32 per (token, kv head)
    const float *v_scale;
    const int *qo_indptr;    // multi-token rows: [B+1] query rows per request (q, out: [total_q, Hq, D]);
                             // null: one row per sequence (a decode group wider than one block)
    size_t total_rows;       // rows of out / lse / the partials: B*Hq, or total_q*Hq
    int q_tiles;             // multi-token rows: blocks per (request, kv head) along its rows
    int total_q, max_q_len;  // multi-token rows: rows of q, and the most rows one request may have
    int causal;              // multi-token rows: row i of a request with n rows and L keys sees keys <= L-n+i
    int B, Hq, Hkv, G, P, log2P, num_pages, max_pages;
    int chunk_tokens, num_splits;
    int box4;                // 1: the tensor maps are 4-D and one box spans all D columns
    int cluster;             // 1 (decode): the S splits of each (b, kv head) are one thread-block
                             // cluster and split 0 merges the partials in its shared memory
    int longest_first;       // 1 (grids of several waves, B <= kLongestFirstMaxB): grid row z
                             // serves the z-th longest sequence
    int adapt_slots;         // > 0 (decode, automatic split count): the keys per split come from
                             // the batch's lengths, about one block per slot (this many) over
                             // its keys; chunk_tokens is then the largest chunk
    int min_chunk;           // the smallest adaptive chunk (a multiple of the stage keys)

    float scale_log2;        // scale * log2(e)
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ void record_status(int *status, int code)
{
    atomicCAS(status, 0, code);
}

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.4426950408889634f;

// Byte offset of 16-byte chunk c (0 .. D/16-1) of row r in one fp8 code tile as the
// TMA box lands it: [box j][column block][box_t rows][INNER bytes] with INNER =
// min(D, 128), swizzled like the TMA's 128B (64B when INNER == 64) mode.
template <int D>
__device__ __forceinline__ uint32_t code_offset(int r, int c, int log2_box_t)
{
    constexpr int INNER = D < 128 ? D : 128;
    constexpr int CB = D / INNER;
    constexpr int CPI = INNER / 16;
    const int cb = c / CPI, cc = c % CPI;
    int row;
    if constexpr (CB == 1) {
        row = r;
    } else {
        const int j = r >> log2_box_t, rr = r & ((1 << log2_box_t) - 1);
        row = ((j * CB + cb) << log2_box_t) + rr;
    }
    const uint32_t lin = (uint32_t)(row * INNER + cc * 16);
    constexpr uint32_t kMask = INNER == 128 ? 7u : 3u;
    return lin ^ (((lin >> 7) & kMask) << 4);
}

// One split's normalised partial output, dims d .. d+3 of block row h: the warps' accumulators
// weighted by their combine factors, summed in warp order.
template <int W, int H8, int RS>
__device__ __forceinline__ float4 block_partial(const float *red, const float *sm_f, int h, int d)
{
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
        const float f = sm_f[w * H8 + h];
        const float *r = red + (w * H8 + h) * RS + d;
        o.x = __fmaf_rn(r[0], f, o.x);
        o.y = __fmaf_rn(r[1], f, o.y);
        o.z = __fmaf_rn(r[2], f, o.z);
        o.w = __fmaf_rn(r[3], f, o.w);
    }
    return o;
}

// The split merge (FlashQuant wiki "CUDA Kernels", split_k_reduce.cu "Algorithm"): per output
// row, split s weighted by exp(lse_s - M), M the largest lse (natural log; -inf marks an empty
// split), the weighted outputs summed in split order and divided by the weight sum.  Taken
// PB splits at a time: the loads of a batch are all issued before any is used (this merge runs
// at the tail of the kernel, where each round trip to memory is long), the batch's largest lse
// joins the running maximum m, and what was summed before is rescaled by exp(m_old - m).  With
// at most PB splits this is the two-pass form exactly.  load(k, s, v, l) gives element k's
// split-s output (4 dims) and lse.  Shared by the workspace merge and the cluster merge, so
// both give the same bits.
template <int NE, int PB, class Load>
__device__ __forceinline__ void merge_splits(int S, Load load, float4 (&a)[NE], float (&m)[NE], float (&wsum)[NE])
{
    const float ninf = -__int_as_float(0x7f800000);
#pragma unroll
    for (int k = 0; k < NE; ++k) {
        a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        m[k] = ninf;
        wsum[k] = 0.f;
    }
    for (int s0 = 0; s0 < S; s0 += PB) {
        float4 v[NE][PB];
        float l[NE][PB];
#pragma unroll
        for (int j = 0; j < PB; ++j)
#pragma unroll
            for (int k = 0; k < NE; ++k) {
                if (s0 + j < S) {
                    load(k, s0 + j, v[k][j], l[k][j]);
                } else {
                    v[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    l[k][j] = ninf;
                }
            }
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            float mb = m[k];
#pragma unroll
            for (int j = 0; j < PB; ++j) mb = fmaxf(mb, l[k][j]);
            const float mr = mb == ninf ? 0.f : mb;  // every split so far empty
            const float f_old = ex2(__fmul_rn(m[k] - mr, kLog2e));
            a[k].x = __fmul_rn(a[k].x, f_old);
            a[k].y = __fmul_rn(a[k].y, f_old);
            a[k].z = __fmul_rn(a[k].z, f_old);
            a[k].w = __fmul_rn(a[k].w, f_old);
            wsum[k] = __fmul_rn(wsum[k], f_old);
#pragma unroll
            for (int j = 0; j < PB; ++j) {
                const float w = ex2(__fmul_rn(l[k][j] - mr, kLog2e));
                a[k].x = __fmaf_rn(v[k][j].x, w, a[k].x);
                a[k].y = __fmaf_rn(v[k][j].y, w, a[k].y);
                a[k].z = __fmaf_rn(v[k][j].z, w, a[k].z);
                a[k].w = __fmaf_rn(v[k][j].w, w, a[k].w);
                wsum[k] = __fadd_rn(wsum[k], w);
            }
            m[k] = mb;
        }
    }
}

// The merged result of one output row's dims d .. d+3: bf16 out, and (d == 0) the natural-log lse.
__device__ __forceinline__ void merge_write(__nv_bfloat16 *out_row, float *lse_row, int d, const float4 a,
                                           const float m, const float wsum)
{
    const float ninf = -__int_as_float(0x7f800000);
    const float inv = m == ninf ? 0.f : 1.f / wsum;
    uint2 packed;
    packed.x = pack_bf16x2(a.x * inv, a.y * inv);
    packed.y = pack_bf16x2(a.z * inv, a.w * inv);
    *reinterpret_cast<uint2 *>(out_row + d) = packed;
    if (d == 0 && lse_row) *lse_row = m == ninf ? ninf : m + __logf(wsum);
}

template <int D, int NT, bool KV8, bool MQ, bool ADAPT>
__global__ void __launch_bounds__(Tiling<D>::W * 32, target_blocks(D, NT, KV8))
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeParams p)
{
    constexpr int T = stage_keys(D, NT, KV8);
    constexpr int W = Tiling<D>::W;
    constexpr int R = ring_depth(D, NT, KV8);
    constexpr int DC = D / 64;            // 128-byte box columns per key row
    constexpr int KS = D / 16;            // k-steps of the score mma, d-tiles of the PV mma
    constexpr int MT = T / 16;            // 16-key mma tiles per stage
    constexpr int H8 = NT * 8;            // padded heads
    constexpr int TILE = KV8 ? T * D : T * D * 2;  // bytes of one K (or V) tile in the ring
    constexpr int STAGE = 2 * TILE;
    constexpr int SUB = T * 128;          // bytes of one 64-dim column block of a tile
    constexpr int RS = D + 4;             // f32 stride of the combine buffer rows

    // kv head fastest: the blocks of one (split, sequence) start together and read the
    // same pages' head slices, which share DRAM rows.  MQ: blockIdx.x also carries the
    // tile qt of the (token, head) rows of the group.
    const int kvh = MQ ? (int)(blockIdx.x % (unsigned)p.Hkv) : (int)blockIdx.x;
    const int qt = MQ ? (int)(blockIdx.x / (unsigned)p.Hkv) : 0;
    const int c = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, cc = lane & 3;
    const int G = p.G;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_addr - raw_addr);
    const SmemLayout lay = smem_layout(D, T, W, R, NT, p.chunk_tokens, p.P, KV8);

    // Cluster merge: each block initialises its two cluster barriers, then every thread
    // arrives on the cluster barrier before any block of the cluster may exit; a block that
    // waits on that barrier later knows every block's barriers are initialised.
    const uint32_t xbar_ready = base_addr + (uint32_t)lay.xbar, xbar_full = xbar_ready + 8u;
    if (!MQ && p.cluster) {
        if (threadIdx.x == 0) {
            mbar_init(xbar_ready, 1);
            mbar_init(xbar_full, 1);
            fence_barrier_init();
        }
        cluster_arrive();
    }

    // Launched with PDL, the block gets here while the previous kernel (say the KV
    // append) may still run: fetch the tensor maps (kernel parameters), then wait for
    // its writes before reading any input.
    if (threadIdx.x == 0) {
        prefetch_tensor_map(&tmK);
        prefetch_tensor_map(&tmV);
        // The block's length and the first lines of its block-table slice into L2 now, so that
        // the table read that depends on the length finds them there.  Safe before the wait: a
        // line the previous kernel writes later is updated in L2, which serves every later read.
        if (!ADAPT && !p.longest_first) {
            prefetch_l2(p.seq_lens + blockIdx.z);
            const long pg = ((long)blockIdx.y * p.chunk_tokens) >> p.log2P;
            const int *row = p.block_table + (size_t)blockIdx.z * p.max_pages;
            if (pg < p.max_pages) prefetch_l2(row + pg);
            if (pg + 32 < p.max_pages) prefetch_l2(row + pg + 32);
        }
    }
    griddep_wait();

    // ---- one pass over the batch's lengths (in the ring, before any copy lands there) ----
    // Which sequence: on grids of several waves grid row z takes the z-th longest sequence (ties
    // by index), so that the blocks of whole chunks start first and the short ones fill the last
    // wave, instead of a long sequence's blocks starting last and running alone at the end.
    // Adaptive split count (decode, automatic split count): the plan sizes the splits for
    // sequences of the table's full width; from the batch's actual lengths every block takes
    // chunks of about (total keys x Hkv / slots) keys, at least min_chunk, at most the planned
    // chunk, and enough that no sequence needs more than the planned splits (Atlas "CUDA Kernel
    // Engineering", "The kernel inventory": adaptive split count).  Every block computes the same
    // value from the same lengths, so the splits of a group agree on their count.  An invalid
    // length counts as empty.
    const int Lmax = p.max_pages * p.P;
    int b = (int)blockIdx.z;
    int chunk = p.chunk_tokens;
    bool have_L = false;
    int L_raw = 0;
    if constexpr (ADAPT) {  // the adaptive instantiation (decode only) always takes this pass
        constexpr bool adapt = !MQ;
        int *lens = reinterpret_cast<int *>(base);        // [B <= 1024] raw lengths (longest first)
        int *pick = reinterpret_cast<int *>(base + 4096);
        int *own = pick + 1;                                // the raw length of sequence blockIdx.z
        long long *wsum = reinterpret_cast<long long *>(base + 4104);
        int *wmax = reinterpret_cast<int *>(base + 4104 + W * 8);
        long long lsum = 0;
        int lmax = 0;
        for (int i = threadIdx.x; i < p.B; i += W * 32) {
            const int li = p.seq_lens[i];
            const int v = (li < 0 || li > Lmax) ? 0 : li;
            if (p.longest_first) lens[i] = li;
            if (i == b) *own = li;
            lsum += v;
            lmax = max(lmax, v);
        }
        __syncthreads();
        if (adapt && !p.longest_first) {
            // A later split that starts past the sequence even at the smallest chunk the rule below
            // can give (min_chunk, or the planned chunk where that is smaller) has nothing to do.
            // It must not leave unless it is empty at the chunk every block computes: split 0 of a
            // cluster signals every non-empty split's shared memory.
            const int own_len = *own, own_v = (own_len < 0 || own_len > Lmax) ? 0 : own_len;
            const int lo = min(p.min_chunk, p.chunk_tokens);
            if (c > 0 && (long long)c * lo >= own_v) return;
        }
        if (adapt) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
                lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            }
            if (lane == 0) {
                wsum[warp] = lsum;
                wmax[warp] = lmax;
            }
            __syncthreads();
            if (threadIdx.x == 0) {  // one thread divides; the others read the result
                lsum = 0;
                lmax = 0;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    lsum += wsum[w];
                    lmax = max(lmax, wmax[w]);
                }
                long long cc = (lsum * p.Hkv + p.adapt_slots - 1) / p.adapt_slots;
                cc = max(cc, (long long)(lmax + p.num_splits - 1) / p.num_splits);
                cc = max(cc, (long long)p.min_chunk);
                cc = (cc + T - 1) / T * T;
                *pick = (int)min(cc, (long long)p.chunk_tokens);
            }
            __syncthreads();
            chunk = *pick;
            __syncthreads();  // pick is reused by the ranking below
        }
        if (p.longest_first) {
            for (int i = threadIdx.x; i < p.B; i += W * 32) {
                const int ri = lens[i], li = (ri < 0 || ri > Lmax) ? 0 : ri;
                int rank = 0;
                for (int j = 0; j < p.B; ++j) {
                    const int rj = lens[j], lj = (rj < 0 || rj > Lmax) ? 0 : rj;
                    rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
                }
                if (rank == (int)blockIdx.z) *pick = i;
            }
            __syncthreads();
            b = *pick;
            L_raw = lens[b];
        } else {
            L_raw = *own;
        }
        have_L = true;
        __syncthreads();  // the ring is free again before the first copies
    } else if (p.longest_first) {
        int *lens = reinterpret_cast<int *>(base);
        int *pick = lens + p.B;
        for (int i = threadIdx.x; i < p.B; i += W * 32) {
            const int li = p.seq_lens[i];
            lens[i] = (li < 0 || li > Lmax) ? 0 : li;  // an invalid length counts as empty
        }
        __syncthreads();
        for (int i = threadIdx.x; i < p.B; i += W * 32) {
            const int li = lens[i];
            int rank = 0;
            for (int j = 0; j < p.B; ++j) {
                const int lj = lens[j];
                rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
            }
            if (rank == (int)blockIdx.z) *pick = i;
        }
        __syncthreads();
        b = *pick;
        __syncthreads();  // the ring is free again before the first copies
    }

    // ---- length, split range ------------------------------------------------
    int L = have_L ? L_raw : p.seq_lens[b];
    if (L < 0 || L > Lmax) {  // invalid length: the sequence is treated as empty
        if (threadIdx.x == 0 && c == 0 && kvh == 0) record_status(p.status, PKV_ERR_BAD_SEQ_LEN);
        L = 0;
    }
    // The block's rows: decode, the G query heads of the group (one query row per
    // sequence); MQ, rows rr = qt*H8 + r of the group's (token i, head h) rows, rr = i*G + h.
    int n_q = 1, q_base = b, row_begin = 0, nrows = G;
    if constexpr (MQ) {
        if (p.qo_indptr) {
            q_base = p.qo_indptr[b];
            n_q = p.qo_indptr[b + 1] - q_base;
            if (q_base < 0 || n_q < 0 || n_q > p.max_q_len || q_base + n_q > p.total_q) {
                // a malformed row range: nothing of this request is read or written
                if (threadIdx.x == 0 && c == 0 && kvh == 0 && qt == 0) record_status(p.status, PKV_ERR_BAD_QO_INDPTR);
                return;
            }
        }  // no qo_indptr: one query row per sequence (a decode group wider than one block)
        row_begin = qt * H8;
        nrows = min(H8, n_q * G - row_begin);
        if (nrows <= 0) return;  // this tile of the group is past the request's rows
    }
    // global row (query row * Hq + query head) of block row r < nrows
    auto grow = [&](int r) -> size_t {
        if constexpr (MQ) {
            const int rr = row_begin + r, i = rr / G;
            return (size_t)(q_base + i) * p.Hq + kvh * G + (rr - i * G);
        } else {
            return (size_t)b * p.Hq + kvh * G + r;
        }
    };
    // MQ with the causal mask: the last key block row r sees (keys past it get -inf)
    auto key_limit = [&](int r) -> int { return (MQ && p.causal) ? L - n_q + (row_begin + r) / G : L - 1; };

    const int tok_begin = c * chunk;
    if (c > 0 && tok_begin >= L) return;  // empty split: the merge never reads it
    if (L == 0) {                          // empty sequence: out = 0, lse = -inf
        for (int i = threadIdx.x; i < nrows * D; i += W * 32)
            p.out[grow(i / D) * D + (i % D)] = __float2bfloat16_rn(0.f);
        if (p.lse)
            for (int i = threadIdx.x; i < nrows; i += W * 32) p.lse[grow(i)] = -__int_as_float(0x7f800000);
        return;
    }
    const int tok_end = min(tok_begin + chunk, L);
    const int n_chunks = (L + chunk - 1) / chunk;
    const int n_stages = (tok_end - tok_begin + T - 1) / T;
    const int page_begin = tok_begin >> p.log2P;
    const int page_end = ((tok_end - 1) >> p.log2P) + 1;
    const int box_t = T < p.P ? T : p.P;   // keys per TMA box (one page slice)
    const int nbox = T / box_t;

    // ---- shared memory ------------------------------------------------------
    const uint32_t ring_addr = base_addr + (uint32_t)lay.ring;
    const uint32_t scale_addr = base_addr + (uint32_t)lay.scales;  // KV8: [W*R][K scales T | V scales T]
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + lay.bars);
    float *sm_m = reinterpret_cast<float *>(base + lay.m);
    float *sm_l = reinterpret_cast<float *>(base + lay.l);
    float *sm_lt = reinterpret_cast<float *>(base + lay.lt);
    float *sm_f = reinterpret_cast<float *>(base + lay.f);
    float *sm_lse = reinterpret_cast<float *>(base + lay.lse);
    int *sm_tab = reinterpret_cast<int *>(base + lay.table);
    float *red = reinterpret_cast<float *>(base);  // reuses the ring after the main loop

    // ---- page ids of this warp's first R stages, one per lane, straight from the block
    // table: the first copies then wait for one table read instead of the whole staging
    constexpr int kMaxBoxes = T / 8;  // boxes per stage at the smallest page size
    int first_id = -1;
    {
        const int r = lane / nbox, j = lane - r * nbox;
        const int s0 = warp + r * W;
        const int t = tok_begin + s0 * T + j * box_t;
        if (r < R && s0 < n_stages && t < tok_end) {
            const int pg = p.block_table[(size_t)b * p.max_pages + (t >> p.log2P)];
            first_id = (unsigned)pg < (unsigned)p.num_pages ? pg : -1;
        }
    }

    // ---- query fragments (B operand of the score mma): q^T[d, head] --------------
    // Loaded early, so that their latency overlaps the first copies and the table staging.
    uint32_t qf[KS][NT][2];
    float score_mul = p.scale_log2;  // KV8: times 2^-eq
    if constexpr (!KV8) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = nt * 8 + g;
            const uint32_t *qp =
                reinterpret_cast<const uint32_t *>(p.q + grow(head < nrows ? head : 0) * D + 2 * cc);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qf[ks][nt][0] = head < nrows ? __ldg(qp + ks * 8) : 0u;
                qf[ks][nt][1] = head < nrows ? __ldg(qp + ks * 8 + 4) : 0u;
            }
        }
    } else {
        // f16, scaled by 2^eq, columns 16ks + 4cc .. +3 in the lane's k slots (see above)
        uint2 raw[KS][NT];
        float qmax = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = nt * 8 + g;
            const uint2 *qp = reinterpret_cast<const uint2 *>(p.q + grow(head < nrows ? head : 0) * D + 4 * cc);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                raw[ks][nt] = head < nrows ? __ldg(qp + ks * 4) : make_uint2(0u, 0u);
                qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(bf16_lo(raw[ks][nt].x)), fabsf(bf16_hi(raw[ks][nt].x))),
                                         fmaxf(fabsf(bf16_lo(raw[ks][nt].y)), fabsf(bf16_hi(raw[ks][nt].y)))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
        const int eq = qmax > 0.f ? max(-126, min(126, 14 - ilog2f(qmax))) : 0;
        const float qs = exp2i(eq);
        score_mul = p.scale_log2 * exp2i(-eq);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint2 r = raw[ks][nt];
                qf[ks][nt][0] = pack_f16x2(bf16_lo(r.x) * qs, bf16_hi(r.x) * qs);
                qf[ks][nt][1] = pack_f16x2(bf16_lo(r.y) * qs, bf16_hi(r.y) * qs);
            }
    }

    // ---- producer: lane 0 of each warp fills that warp's ring ----------------
    const uint64_t policy = l2_policy_evict_first();
    // Copies of stage s into ring slot `slot`; ids[j] is the page of box j (-1: not loaded).
    auto issue_ids = [&](int s, int slot, const int (&ids)[kMaxBoxes]) {
        const int t0 = tok_begin + s * T;
        const uint32_t bar = smem_addr(&bars[warp * R + slot]);
        const uint32_t kdst = ring_addr + (uint32_t)((warp * R + slot) * STAGE);
        constexpr uint32_t kBoxBytes = KV8 ? 2u * (uint32_t)D + 8u : 2u * DC * 128u;  // per key row: K, V (+ scales)
        uint32_t bytes = 0;
#pragma unroll
        for (int j = 0; j < kMaxBoxes; ++j)
            if (j < nbox && ids[j] >= 0) bytes += kBoxBytes * box_t;
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int j = 0; j < kMaxBoxes; ++j) {
            if (j >= nbox || ids[j] < 0) continue;
            const int pg = ids[j];
            const int t = t0 + j * box_t;
            const int slot_in_page = t & (p.P - 1);
            const int row = pg * p.P + slot_in_page;
            if constexpr (KV8) {
                // codes: one (INNER bytes, box_t rows, D/INNER column blocks, 1 head) box per
                // tensor; scales: box_t contiguous f32 of this head's slice of the page
                const uint32_t off = (uint32_t)(j * box_t * D);
                tma_load_4d(kdst + off, &tmK, 0, row, 0, kvh, bar, policy);
                tma_load_4d(kdst + TILE + off, &tmV, 0, row, 0, kvh, bar, policy);
                const size_t sidx = ((size_t)pg * p.Hkv + kvh) * p.P + slot_in_page;
                const uint32_t sdst = scale_addr + (uint32_t)((warp * R + slot) * (2 * T * 4) + j * box_t * 4);
                bulk_copy_g2s(sdst, p.k_scale + sidx, (uint32_t)box_t * 4u, bar);
                bulk_copy_g2s(sdst + T * 4, p.v_scale + sidx, (uint32_t)box_t * 4u, bar);
            } else if (p.box4 && nbox == 1) {
                // one box per tensor: (64 dims, box_t rows, all D/64 column blocks, 1 head)
                tma_load_4d(kdst, &tmK, 0, row, 0, kvh, bar, policy);
                tma_load_4d(kdst + TILE, &tmV, 0, row, 0, kvh, bar, policy);
            } else {
#pragma unroll
                for (int dc = 0; dc < DC; ++dc) {
                    const uint32_t off = (uint32_t)(dc * SUB + j * box_t * 128);
                    tma_load_3d(kdst + off, &tmK, dc * 64, kvh, row, bar, policy);
                    tma_load_3d(kdst + TILE + off, &tmV, dc * 64, kvh, row, bar, policy);
                }
            }
        }
    };
    // Later stages take their page ids from the staged table slice.
    auto issue = [&](int s, int slot) {
        int ids[kMaxBoxes];
#pragma unroll
        for (int j = 0; j < kMaxBoxes; ++j) {
            const int t = tok_begin + s * T + j * box_t;
            ids[j] = (j < nbox && t < tok_end) ? sm_tab[(t >> p.log2P) - page_begin] : -1;
        }
        issue_ids(s, slot, ids);
    };

    // Lane 0 of each warp initialises the warp's own barriers and issues its first R stages.
    {
        int ids[R][kMaxBoxes];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int j = 0; j < kMaxBoxes; ++j) {
                const int v = __shfl_sync(0xffffffffu, first_id, (r * nbox + j) & 31);
                ids[r][j] = j < nbox ? v : -1;
            }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) mbar_init(smem_addr(&bars[warp * R + r]), 1);
            fence_barrier_init();
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int s0 = warp + r * W;
                if (s0 < n_stages) issue_ids(s0, r, ids[r]);
            }
        }
    }

    // Stage this split's block-table slice for the later stages; out-of-range ids become -1.
    int bad = 0;
    for (int i = threadIdx.x; i < page_end - page_begin; i += W * 32) {
        int pg = p.block_table[(size_t)b * p.max_pages + page_begin + i];
        if ((unsigned)pg >= (unsigned)p.num_pages) {
            record_status(p.status, PKV_ERR_BAD_PAGE_INDEX);
            pg = -1;
            bad = 1;
        }
        sm_tab[i] = pg;
    }
    const bool any_bad = __syncthreads_or(bad) != 0;

    // ---- consumer state -----------------------------------------------------
    float acc[KS][NT][4];
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;
    float m_run[NT][2], l_run[NT][2], lt_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -__int_as_float(0x7f800000);
        l_run[nt][0] = l_run[nt][1] = 0.f;
        lt_run[nt][0] = lt_run[nt][1] = 0.f;
    }

    // MQ: the key limit of each of this lane's score columns (rows nt*8 + 2cc + j), and the
    // first key some row of the block must not see (stages from there on take the masked body)
    int klim[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = nt * 8 + 2 * cc + j;
            klim[nt][j] = r < nrows ? key_limit(r) : L - 1;
        }
    const int causal_from = key_limit(0) + 1;

    auto key_valid = [&](int t) -> bool {
        return t < tok_end && sm_tab[(t >> p.log2P) - page_begin] >= 0;
    };

    int ev_run = -126;  // KV8: running maximum of this warp's V-scale exponents
    // KV8: per-lane ldmatrix offsets within a code tile (the same for K and V and for every
    // stage): matrix (lane >> 3) of each x4 load covers keys 0-7 / 8-15 of chunks 2kp, 2kp+1
    uint32_t coff[MT][KS / 2];
    if constexpr (KV8) {
        const int log2_box_t = box_t == 8 ? 3 : box_t == 16 ? 4 : 5;  // used for D = 256 only
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp)
                coff[mt][kp] = code_offset<D>(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * kp + (lane >> 4),
                                              log2_box_t);
    }

    // One stage of T keys; MASKED (a compile-time flag) adds the key-validity checks that
    // only the stages holding a split's tail, or a bad page, need.
    auto run_stage = [&](auto masked_tag, const int t0, const uint32_t kbase, const int slot) {
        constexpr bool MASKED = decltype(masked_tag)::value;
        const uint32_t vbase = kbase + TILE;

        // S^T = K q^T; with few independent tiles the k steps alternate between two
        // accumulators (two shorter mma chains), otherwise the tiles give the parallelism
        constexpr bool kTwoChains = MT * NT <= 2;
        float sc[MT][NT][4], sc2[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[mt][nt][e] = sc2[mt][nt][e] = 0.f;
        if constexpr (!KV8) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int chunk = (ks & 3) * 2 + (lane >> 4);
                    const uint32_t addr = kbase + (uint32_t)((ks >> 2) * SUB + row * 128 + ((chunk ^ (row & 7)) << 4));
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816((kTwoChains && (ks & 1)) ? sc2[mt][nt] : sc[mt][nt], a0, a1, a2, a3,
                                       qf[ks][nt][0], qf[ks][nt][1]);
                }
            }
        } else {
            // each register of an x4 load holds a lane's 4 codes of one chunk: the low pair
            // goes to k slots 2t, 2t+1, the high pair to 2t+8, 2t+9
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4(kbase + coff[mt][kp], r0, r1, r2, r3);
                    uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                    e4m3x4_to_f16x2x2(r0, a0, a2);
                    e4m3x4_to_f16x2x2(r1, a1, a3);
                    e4m3x4_to_f16x2x2(r2, c0, c2);
                    e4m3x4_to_f16x2x2(r3, c1, c3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16_16816(sc[mt][nt], a0, a1, a2, a3, qf[2 * kp][nt][0], qf[2 * kp][nt][1]);
                        mma_f16_16816(kTwoChains ? sc2[mt][nt] : sc[mt][nt], c0, c1, c2, c3, qf[2 * kp + 1][nt][0],
                                      qf[2 * kp + 1][nt][1]);
                    }
                }
            }
        }

        // scale to log2 units (KV8: times the key's scale), mask, running max
        float kmul[MT][2], vmul[MT][2];
        float vfac = 1.f;  // KV8: rescale of the accumulators when the V-scale exponent rises
        if constexpr (KV8) {
            const uint32_t sb = scale_addr + (uint32_t)((warp * R + slot) * (2 * T * 4));
            // the stage's largest V-scale exponent: the exponent of the largest |scale| bit
            // pattern (non-negative floats order as their bits), over the valid keys
            uint32_t vbits = 0u;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = mt * 16 + g + 8 * h;
                    kmul[mt][h] = ld_shared_f32(sb + (uint32_t)r * 4u) * score_mul;
                    vmul[mt][h] = ld_shared_f32(sb + (uint32_t)(T + r) * 4u);
                    if (MASKED && !key_valid(t0 + r)) vmul[mt][h] = 0.f;
                    vbits = max(vbits, __float_as_uint(vmul[mt][h]) & 0x7fffffffu);
                }
            const int ev = min(126, ilog2f(__uint_as_float(__reduce_max_sync(0xffffffffu, vbits))));
            if (ev > ev_run) {
                vfac = exp2i(ev_run - ev);
                ev_run = ev;
            }
            const float inv = exp2i(-ev_run);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                vmul[mt][0] *= inv;
                vmul[mt][1] *= inv;
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) kmul[mt][0] = kmul[mt][1] = vmul[mt][0] = vmul[mt][1] = p.scale_log2;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float v = (kTwoChains ? sc[mt][nt][e] + sc2[mt][nt][e] : sc[mt][nt][e]) * kmul[mt][e >> 1];
                    if (MASKED) {
                        const int t = t0 + mt * 16 + g + ((e >> 1) << 3);
                        if (!key_valid(t) || (MQ && t > klim[nt][e & 1])) v = -__int_as_float(0x7f800000);
                    }
                    sc[mt][nt][e] = v;
                }
        float alpha[NT][2], mref[NT][2];
        bool rescale = vfac != 1.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float mx = -__int_as_float(0x7f800000);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) mx = fmaxf(mx, fmaxf(sc[mt][nt][h2], sc[mt][nt][h2 + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float m_new = fmaxf(m_run[nt][h2], mx);
                const float r = (m_new == -__int_as_float(0x7f800000)) ? 0.f : m_new;
                alpha[nt][h2] = ex2(m_run[nt][h2] - r);
                mref[nt][h2] = r;
                m_run[nt][h2] = m_new;
                l_run[nt][h2] *= alpha[nt][h2];
                lt_run[nt][h2] *= alpha[nt][h2];
                rescale |= alpha[nt][h2] != 1.f;
            }
        // the accumulators change only when a running maximum moved (multiplying by 1 is exact)
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float f0 = alpha[nt][0] * vfac, f1 = alpha[nt][1] * vfac;
#pragma unroll
                for (int i = 0; i < KS; ++i) {
                    acc[i][nt][0] *= f0;
                    acc[i][nt][1] *= f1;
                    acc[i][nt][2] *= f0;
                    acc[i][nt][3] *= f1;
                }
            }
        }

        // O^T += V^T P^T, one 16-key tile at a time
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float p0 = ex2(sc[mt][nt][0] - mref[nt][0]), p1 = ex2(sc[mt][nt][1] - mref[nt][1]);
                const float p2 = ex2(sc[mt][nt][2] - mref[nt][0]), p3 = ex2(sc[mt][nt][3] - mref[nt][1]);
                l_run[nt][0] += p0 + p2;
                l_run[nt][1] += p1 + p3;
                uint32_t x0, x1;
                if constexpr (KV8) {
                    x0 = pack_f16x2(p0 * vmul[mt][0], p1 * vmul[mt][0]);
                    x1 = pack_f16x2(p2 * vmul[mt][1], p3 * vmul[mt][1]);
                } else {
                    x0 = pack_bf16x2(p0, p1);
                    x1 = pack_bf16x2(p2, p3);
                    lt_run[nt][0] += bf16_lo(x0) + bf16_lo(x1);
                    lt_run[nt][1] += bf16_hi(x0) + bf16_hi(x1);
                }
                pb[nt][0] = movmatrix_trans(x0);
                pb[nt][1] = movmatrix_trans(x1);
            }
            // invalid keys' V values are zeroed in registers (their probability is 0, and 0 * NaN is NaN)
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (MASKED) {
                const int t = t0 + mt * 16 + 2 * cc;
                vm0 = (key_valid(t) ? 0x0000ffffu : 0u) | (key_valid(t + 1) ? 0xffff0000u : 0u);
                vm1 = (key_valid(t + 8) ? 0x0000ffffu : 0u) | (key_valid(t + 9) ? 0xffff0000u : 0u);
            }
            if constexpr (!KV8) {
#pragma unroll
                for (int md = 0; md < KS; ++md) {
                    const int row = mt * 16 + (lane & 7) + (lane >> 4) * 8;
                    const int chunk = (md & 3) * 2 + ((lane >> 3) & 1);
                    const uint32_t addr = vbase + (uint32_t)((md >> 2) * SUB + row * 128 + ((chunk ^ (row & 7)) << 4));
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(addr, a0, a1, a2, a3);
                    if (MASKED) {
                        a0 &= vm0;
                        a1 &= vm0;
                        a2 &= vm1;
                        a3 &= vm1;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[md][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
            } else {
                // ldmatrix.trans of the code bytes: a register holds keys (2t, 2t+1) x dims
                // (2g, 2g+1) of a 16-dim chunk; the byte permute pairs the keys per dim, so
                // PV rows g, g+8 are dims 2g, 2g+1 of the chunk
#pragma unroll
                for (int mp = 0; mp < KS / 2; ++mp) {
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4_trans(vbase + coff[mt][mp], r0, r1, r2, r3);
                    uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                    e4m3x4_to_f16x2x2(__byte_perm(r0, 0u, 0x3120), a0, a1);
                    e4m3x4_to_f16x2x2(__byte_perm(r1, 0u, 0x3120), a2, a3);
                    e4m3x4_to_f16x2x2(__byte_perm(r2, 0u, 0x3120), c0, c1);
                    e4m3x4_to_f16x2x2(__byte_perm(r3, 0u, 0x3120), c2, c3);
                    if (MASKED) {
                        a0 &= vm0;
                        a1 &= vm0;
                        a2 &= vm1;
                        a3 &= vm1;
                        c0 &= vm0;
                        c1 &= vm0;
                        c2 &= vm1;
                        c3 &= vm1;
                    }
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16_16816(acc[2 * mp][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                        mma_f16_16816(acc[2 * mp + 1][nt], c0, c1, c2, c3, pb[nt][0], pb[nt][1]);
                    }
                }
            }
        }
    };

    int failed_it = -1;
    for (int it = 0;; ++it) {
        const int s = warp + it * W;
        if (s >= n_stages) break;
        const int slot = it % R;
        const uint32_t parity = (uint32_t)((it / R) & 1);
        const bool ok = mbar_wait_bounded(smem_addr(&bars[warp * R + slot]), parity, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT);
            failed_it = it;
            break;
        }
        const int t0 = tok_begin + s * T;
        const uint32_t kbase = ring_addr + (uint32_t)((warp * R + slot) * STAGE);
        if ((t0 + T > tok_end) || any_bad || (MQ && t0 + T > causal_from))
            run_stage(std::true_type{}, t0, kbase, slot);
        else
            run_stage(std::false_type{}, t0, kbase, slot);

        __syncwarp();
        if (lane == 0) {
            const int ns = s + R * W;
            if (ns < n_stages) issue(ns, slot);
        }
    }
    if (failed_it >= 0) {
        // A copy outlasted its limit.  The warp's later stages (up to R - 1 of them) were issued
        // too: wait for each, bounded, so that none lands in shared memory after the block has
        // exited unless it also outlasts the limit.
        for (int it = failed_it + 1; it < failed_it + R && warp + it * W < n_stages; ++it)
            mbar_wait_bounded(smem_addr(&bars[warp * R + it % R]), (uint32_t)((it / R) & 1), p.wait_limit_ns);
    }

    griddep_launch_dependents();  // streaming done: the next kernel may start launching

    if constexpr (KV8) {  // back to value units; the f32 denominator normalises
        const float f = exp2i(ev_run);
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][nt][e] *= f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) lt_run[nt][0] = l_run[nt][0], lt_run[nt][1] = l_run[nt][1];
    }

    // ---- per-warp finalisation: reduce the denominators over the key rows ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float l = l_run[nt][h2], lt = lt_run[nt][h2];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            lt += __shfl_xor_sync(0xffffffffu, lt, 4);
            lt += __shfl_xor_sync(0xffffffffu, lt, 8);
            lt += __shfl_xor_sync(0xffffffffu, lt, 16);
            l_run[nt][h2] = l;
            lt_run[nt][h2] = lt;
        }
    __syncthreads();  // every warp is done with the ring: reuse it as the combine buffer
    const bool cl = !MQ && p.cluster && n_chunks > 1;
    if (cl) {
        cluster_wait();  // every block of the cluster has initialised its barriers
        if (c == 0 && threadIdx.x == 0) {
            // split 0's ring past the combine buffer is free: it takes the partials of splits
            // 1 .. n_chunks-1, nrows x (D + 1) f32 each (outputs, then lse)
            mbar_arrive_expect_tx(xbar_full, (uint32_t)((n_chunks - 1) * nrows * (D + 1) * 4));
            for (int r = 1; r < n_chunks; ++r) mbar_arrive_remote(map_to_rank(xbar_ready, (uint32_t)r));
        }
    }
    if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                sm_m[warp * H8 + nt * 8 + 2 * cc + h2] = m_run[nt][h2];
                sm_l[warp * H8 + nt * 8 + 2 * cc + h2] = l_run[nt][h2];
                sm_lt[warp * H8 + nt * 8 + 2 * cc + h2] = lt_run[nt][h2];
            }
    }
#pragma unroll
    for (int md = 0; md < KS; ++md)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // PV rows g, g+8 are dims g, g+8 of the chunk (bf16) or 2g, 2g+1 (fp8)
            const int h0 = nt * 8 + 2 * cc;
            const int d0 = KV8 ? md * 16 + 2 * g : md * 16 + g, d1 = KV8 ? d0 + 1 : d0 + 8;
            float *r0 = red + (warp * H8 + h0) * RS;
            r0[d0] = acc[md][nt][0];
            r0[RS + d0] = acc[md][nt][1];
            r0[d1] = acc[md][nt][2];
            r0[RS + d1] = acc[md][nt][3];
        }
    __syncthreads();

    // ---- block combine: per-head factors, then the outputs ------------------
    if (threadIdx.x < H8) {
        const int h = threadIdx.x;
        float M = -__int_as_float(0x7f800000);
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, sm_m[w * H8 + h]);
        if (M == -__int_as_float(0x7f800000)) {
#pragma unroll
            for (int w = 0; w < W; ++w) sm_f[w * H8 + h] = 0.f;
            sm_lse[h] = -__int_as_float(0x7f800000);
        } else {
            float lsum = 0.f, ltsum = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float e = ex2(sm_m[w * H8 + h] - M);
                lsum += sm_l[w * H8 + h] * e;
                ltsum += sm_lt[w * H8 + h] * e;
            }
            const float inv = 1.f / ltsum;
#pragma unroll
            for (int w = 0; w < W; ++w) sm_f[w * H8 + h] = ex2(sm_m[w * H8 + h] - M) * inv;
            sm_lse[h] = (M + __log2f(lsum)) * kLn2;
        }
    }
    __syncthreads();

    const bool direct = (n_chunks == 1);
    if (direct) {  // the only split of this sequence: final bf16 output and lse
        for (int i = threadIdx.x; i < nrows * D / 2; i += W * 32) {
            const int h = (2 * i) / D, d = 2 * i - h * D;
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float f = sm_f[w * H8 + h];
                o0 += red[(w * H8 + h) * RS + d] * f;
                o1 += red[(w * H8 + h) * RS + d + 1] * f;
            }
            const size_t row = grow(h);
            *reinterpret_cast<uint32_t *>(p.out + row * D + d) = pack_bf16x2(o0, o1);
        }
        if (threadIdx.x < nrows && p.lse) p.lse[grow(threadIdx.x)] = sm_lse[threadIdx.x];
        return;
    }

    // ---- several splits, merged inside the cluster: split 0 holds the partials ----
    if (cl) {
        const uint32_t recv = base_addr + (uint32_t)lay.recv;
        if (c > 0) {
            // wait (bounded: longer than split 0 can take to stream and signal) until split 0's
            // ring is free, then store this split's partial there; the stores complete on split
            // 0's "full" barrier
            if (!mbar_wait_bounded_cluster(xbar_ready, 0, p.wait_limit_ns * (R + 2))) {
                if (threadIdx.x == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT);
                return;
            }
            const uint32_t dst = map_to_rank(recv + (uint32_t)((c - 1) * lay.recv_slot), 0u);
            const uint32_t bar = map_to_rank(xbar_full, 0u);
            for (int i = threadIdx.x; i < nrows * D / 4; i += W * 32) {
                const int h = (4 * i) / D, d = 4 * i - h * D;
                st_async_v4(dst + (uint32_t)((h * D + d) * 4), block_partial<W, H8, RS>(red, sm_f, h, d), bar);
            }
            if (threadIdx.x < nrows)
                st_async_f32(dst + (uint32_t)((H8 * D + threadIdx.x) * 4), sm_lse[threadIdx.x], bar);
            return;
        }
        // split 0: its own partial and the others', merged in split order
        if (!mbar_wait_bounded_cluster(xbar_full, 0, p.wait_limit_ns * (R + 3)) && threadIdx.x == 0)
            record_status(p.status, PKV_ERR_DEVICE_TIMEOUT);
        for (int i = threadIdx.x; i < nrows * D / 4; i += W * 32) {
            const int h = (4 * i) / D, d = 4 * i - h * D;
            float4 a[1];
            float m[1], wsum[1];
            merge_splits<1, kMaxClusterSplits>(
                n_chunks,
                [&](int, int sidx, float4 &v, float &l) {
                    if (sidx == 0) {
                        v = block_partial<W, H8, RS>(red, sm_f, h, d);
                        l = sm_lse[h];
                    } else {
                        const float *slot =
                            reinterpret_cast<const float *>(base + lay.recv + (sidx - 1) * lay.recv_slot);
                        v = *reinterpret_cast<const float4 *>(slot + h * D + d);
                        l = slot[H8 * D + h];
                    }
                },
                a, m, wsum);
            merge_write(p.out + grow(h) * D, p.lse ? p.lse + grow(h) : nullptr, d, a[0], m[0], wsum[0]);
        }
        return;
    }

    // ---- one of several splits: write this split's normalised output and lse ----
    const size_t rows = p.total_rows;
    for (int i = threadIdx.x; i < nrows * D / 4; i += W * 32) {
        const int h = (4 * i) / D, d = 4 * i - h * D;
        *reinterpret_cast<float4 *>(p.part_out + ((size_t)c * rows + grow(h)) * D + d) =
            block_partial<W, H8, RS>(red, sm_f, h, d);
    }
    if (threadIdx.x < nrows) p.part_lse[(size_t)c * rows + grow(threadIdx.x)] = sm_lse[threadIdx.x];

    // ---- the last split of this (b, kv head) to finish merges all of them ----------
    // atomicInc wraps the per-group counter back to 0 on the last arrival, ready for the
    // next call.  The splits are combined in index order whichever block arrives last, so
    // the result does not depend on scheduling.
    __threadfence();
    __syncthreads();
    int *flag = reinterpret_cast<int *>(base + lay.flag);
    if (threadIdx.x == 0)
        *flag = atomicInc(reinterpret_cast<unsigned *>(p.counters + ((size_t)b * p.q_tiles + qt) * p.Hkv + kvh),
                          (unsigned)(n_chunks - 1)) ==
                (unsigned)(n_chunks - 1);
    __syncthreads();
    if (!*flag) return;
    __threadfence();

    constexpr int V4 = D / 4;
    constexpr int NE = 2;
    const int nvec = nrows * V4;
    for (int e0 = threadIdx.x; e0 < nvec; e0 += NE * W * 32) {
        const float *lp[NE];
        const float4 *op[NE];
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int e = e0 + k * W * 32;
            const int h = (e < nvec ? e : 0) / V4, d4 = (e < nvec ? e : 0) - h * V4;
            lp[k] = p.part_lse + grow(h);
            op[k] = reinterpret_cast<const float4 *>(p.part_out + grow(h) * D) + d4;
        }
        float4 a[NE];
        float m[NE], wsum[NE];
        merge_splits<NE, 8>(
            n_chunks,
            [&](int k, int sidx, float4 &v, float &l) {
                v = __ldcg(op[k] + (size_t)sidx * rows * V4);
                l = __ldcg(lp[k] + (size_t)sidx * rows);
            },
            a, m, wsum);
#pragma unroll
        for (int k = 0; k < NE; ++k) {
            const int e = e0 + k * W * 32;
            if (e >= nvec) continue;
            const int h = e / V4, d4 = e - h * V4;
            merge_write(p.out + grow(h) * D, p.lse ? p.lse + grow(h) : nullptr, 4 * d4, a[k], m[k], wsum[k]);
        }
    }
}

}  // namespace pkv
