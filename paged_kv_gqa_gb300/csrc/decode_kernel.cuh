// decode_kernel.cuh -- balanced persistent split-KV paged GQA decode kernel for sm_103a.
//
// Work partition.  Every (sequence b, kv head) pair is a segment of
// ceil(L_b / T) tiles of T keys; laid end to end (kv head by kv head, then
// sequence by sequence), the segments of the batch form one list of tiles,
// and block i of the grid (one block per SM) takes the i-th equal slice of it: ceil(total / grid) tiles, but never fewer than
// a minimum that keeps the partial results rare.  A block therefore streams
// the same number of bytes as every other block whatever the mix of lengths,
// and a long sequence is spread over as many SMs as its share of the batch
// needs.  This is the split-KV ("flash-decoding") scheme with the split points
// chosen from seq_len and the SM count on the device, deterministically
// (FlashQuant wiki "CUDA Kernels", paged_decode.cu: a sequence's key range is
// split over several blocks and the partial softmax states are merged; OASR
// "Kernel Layer", "Fused attention": the split is a pure function of shape and
// SM count, here of the lengths and the SM count).  Each block serves all G =
// Hq/Hkv query heads that read a kv head, so every K/V byte leaves HBM once
// per call (AstrAI "CUDA Kernels", "Q Scheduling and KV Addressing": packing
// the query heads of a group into one block streams K/V once per block).
//
// Warp roles.  Warp W (the item warp) walks the block's slice: each piece of
// a segment that the slice covers is cut into work items of at most
// max_item_tiles tiles; for each item the warp copies the item's block-table
// slice into shared memory (one coalesced warp load per 32 pages, every page
// id checked against the pool) and stages the item's query rows with one bulk
// copy, QS items ahead of use.  Warps 0..W-1 (the consumers) take an item's
// stages round-robin; each consumer warp issues the TMA copies of its own
// stages into its own ring of R stages, R stages ahead of use and on into the
// next items, so eight warps keep copies in flight and HBM does not idle on a
// piece's epilogue.  A stage is T keys of one kv head; the tensor maps view
// k_cache/v_cache as [num_pages*P rows, Hkv, D] and one box is (64 dims, 1
// head, min(T,P) rows), so a copy moves a page slice with no per-thread
// address arithmetic.  The physical row of key j is
// block_table[b][j >> log2 P] * P + (j & (P-1)) (FlashQuant wiki "CUDA
// Kernels", paged_decode.cu "Page Table Addressing").  Boxes land
// 128B-swizzled so the ldmatrix reads below are free of bank conflicts.
//
// Math.  Keys sit on the mma M dimension and the query heads of the group on N
// (8 per tile, padded), so G = 4, 8, 16 map onto m16n8k16 tiles without wasted
// rows:
//     S^T[key, head]  = K[key, :] . q^T[:, head]            (K via ldmatrix, q in registers)
//     O^T[d, head]   += V^T[d, key] . P^T[key, head]        (V via ldmatrix.trans)
// P^T comes out of the S accumulators as bf16 pairs and becomes the B operand
// through movmatrix.trans.  The softmax is the online recurrence in base 2
// (FlashQuant wiki "CUDA Kernels", flash_attention.cu "Online Softmax" and the
// "exp2/log2(e) prescaling" row of its optimisation summary): scores are
// scaled by scale*log2(e) in f32, the running max m, the denominators and the
// accumulators are f32, and each exponential is one ex2.approx.  Row maxima use
// warp shuffles; denominators are summed per thread and reduced once per piece.
// Two denominators are kept: the sum of the f32 probabilities, which gives the
// LSE, and the sum of the bf16-rounded probabilities the PV product uses, which
// normalises the output so it is a convex combination of V rows up to f32
// rounding (a constant V comes back unchanged).
//
// Masking.  Keys at or past L_b (the padded tail of the last page) and keys of
// a page whose id is out of range get score -inf, and their V values are zeroed
// in registers before the PV mma, so NaN or Inf left in unused slots never
// reaches the result (0 * NaN would).
//
// Epilogue.  At the end of a piece the consumer warps merge their states
// pairwise through shared memory into warp 0.  A piece that is a whole segment
// gets its bf16 output and natural-log LSE written directly.  A piece that is
// part of a segment writes its normalised f32 output and LSE to one of the
// block's two partial slots (FlashQuant wiki "CUDA Kernels", paged_decode.cu
// "Partial Output"; here normalised and in natural log), and the block that
// finishes the segment's last piece merges its pieces, in block order, in the
// same launch (split_k_reduce.cu "Algorithm").  Sequences of length 0 get out
// = 0 and lse = -inf.
//
// Failure handling.  Every wait is bounded.  A wait that runs out records
// PKV_ERR_DEVICE_TIMEOUT in the status word and sets a block-wide abort flag,
// after which no wait blocks again, so the kernel always finishes.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "plan.h"
#include "ptx.cuh"

namespace pkv {

struct DecodeParams {
    const __nv_bfloat16 *q;  // [B, Hq, D]
    const int *block_table;  // [B, max_pages]
    const int *seq_lens;     // [B]
    __nv_bfloat16 *out;      // [B, Hq, D]
    float *lse;              // [B, Hq] or nullptr
    float *part_lse;         // [2 * grid, G]     partial slots: two per block
    float *part_out;         // [2 * grid, G, D]
    int *counters;           // [B, Hkv] pieces finished per segment (wraps to 0 after the last)
    int *status;             // workspace status word
    int B, Hq, Hkv, G, P, log2P, num_pages, max_pages;
    int box4;                // 1: the tensor maps are 4-D and one box spans all D columns
    int min_range_tiles;     // lower bound on the tiles of one block's slice
    int max_item_tiles;      // tiles per work item (bounds its block-table slice)
    float scale_log2;        // scale * log2(e)
    unsigned long long wait_limit_ns;
};

__device__ __forceinline__ void record_status(int *status, int code) { atomicCAS(status, 0, code); }

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kFirst = 1, kLast = 2, kEnd = 4;  // ItemDesc::flags

// Work-item descriptor, written by the item warp, read by the consumer warps.
struct ItemDesc {
    int b, kvh, L, tok_begin;          // segment, its length, first key of the item
    int tok_end, page_begin, any_bad, flags;
    int n_pieces, slot, merge_f, merge_f_tail;  // piece merge: count, own partial slot, first block
};

// Named barrier among the consumer warps only (the item warp never joins).
__device__ __forceinline__ void consumer_sync(int nthreads)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Bounded waits with a block-wide abort flag: once one wait has run out, the
// others give up at once, so a stalled copy cannot hold the kernel for long.
struct Waiter {
    volatile int *abort;
    int *status;
    unsigned long long limit_ns;
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const
    {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
        *abort = 1;
        record_status(status, PKV_ERR_DEVICE_TIMEOUT);
        return false;
    }
};

// Partial slot that block j used for its piece of a segment whose first block is f.
__device__ __forceinline__ int piece_slot(const ItemDesc &d, int j)
{
    return 2 * j + (j == d.merge_f ? d.merge_f_tail : 0);
}

// Log-sum-exp merge of the pieces of one (b, kv head) segment, run by the
// consumer warps of the block that finished the segment's last piece.  The
// weight of piece s is exp(lse_s - max_s lse_s); pieces are summed in block
// order, so the result does not depend on which block merges.
template <int D, int W>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, const ItemDesc &d, size_t row0, float *mh,
                                             float *lh, int lane, int warp)
{
    constexpr int CT = W * 32;
    const float ninf = -__int_as_float(0x7f800000);
    const int G = p.G, n = d.n_pieces;
    for (int h = warp; h < G; h += W) {  // per-head max and weight sum over the pieces
        float mx = ninf;
        for (int s = lane; s < n; s += 32) mx = fmaxf(mx, __ldcg(p.part_lse + piece_slot(d, d.merge_f + s) * G + h));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float wsum = 0.f;
        if (mx != ninf)
            for (int s = lane; s < n; s += 32)
                wsum += ex2((__ldcg(p.part_lse + piece_slot(d, d.merge_f + s) * G + h) - mx) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        if (lane == 0) {
            mh[h] = mx;
            lh[h] = wsum;
        }
    }
    consumer_sync(CT);
    constexpr int V4 = D / 4;
    for (int e = threadIdx.x; e < G * V4; e += CT) {
        const int h = e / V4, d4 = e - h * V4;
        const float mx = mh[h];
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        float inv = 0.f;
        if (mx != ninf) {
#pragma unroll 4
            for (int s = 0; s < n; ++s) {
                const int sl = piece_slot(d, d.merge_f + s);
                const float w = ex2((__ldcg(p.part_lse + sl * G + h) - mx) * kLog2e);
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part_out + ((size_t)sl * G + h) * D) + d4);
                a.x += w * v.x;
                a.y += w * v.y;
                a.z += w * v.z;
                a.w += w * v.w;
            }
            inv = 1.f / lh[h];
        }
        uint2 packed;
        packed.x = pack_bf16x2(a.x * inv, a.y * inv);
        packed.y = pack_bf16x2(a.z * inv, a.w * inv);
        *reinterpret_cast<uint2 *>(p.out + (row0 + h) * D + 4 * d4) = packed;
    }
    if (threadIdx.x < G && p.lse) {
        const float mx = mh[threadIdx.x];
        p.lse[row0 + threadIdx.x] = mx == ninf ? ninf : mx + __logf(lh[threadIdx.x]);
    }
}

template <int D, int NT>
__global__ void __launch_bounds__((PTiling<D, NT>::W + 1) * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    using TL = PTiling<D, NT>;
    constexpr int T = TL::T;              // keys per stage (one tile)
    constexpr int W = TL::W;              // consumer warps
    constexpr int R = TL::R;              // stages in flight per consumer warp
    constexpr int QS = TL::QS;            // work-item slots
    constexpr int NTHR = (W + 1) * 32;
    constexpr int CT = W * 32;            // consumer threads
    constexpr int DC = D / 64;            // 128-byte box columns per key row
    constexpr int KS = D / 16;            // k-steps of the score mma, d-tiles of the PV mma
    constexpr int MT = T / 16;            // 16-key mma tiles per stage
    constexpr int H8 = NT * 8;            // padded heads
    constexpr int TILE = T * D * 2;       // bytes of one K (or V) stage tile
    constexpr int STAGE = 2 * TILE;
    constexpr int SUB = T * 128;          // bytes of one 64-dim column block of a tile
    constexpr PersistLayout lay = persist_layout<D, NT>();
    static_assert(R >= 2, "at least two stages in flight per consumer warp");
    static_assert(sizeof(ItemDesc) == kDescBytes, "descriptor size");
    const float ninf = -__int_as_float(0x7f800000);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    const int box_t = T < p.P ? T : p.P;  // keys per TMA box (one page slice)
    const int nbox = T / box_t;           // boxes per stage (1, or T/P when pages are short)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_addr - raw_addr);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + lay.full);
    uint64_t *item_full = reinterpret_cast<uint64_t *>(base + lay.item_full);
    uint64_t *item_empty = reinterpret_cast<uint64_t *>(base + lay.item_empty);
    ItemDesc *desc = reinterpret_cast<ItemDesc *>(base + lay.desc);
    int *tab = reinterpret_cast<int *>(base + lay.tab);
    int *prefix = reinterpret_cast<int *>(base + lay.prefix);  // tiles before each sequence
    float *red = reinterpret_cast<float *>(base + lay.red);    // pairwise-combine buffer
    float *mh = reinterpret_cast<float *>(base + lay.mh);      // merge: per-head max
    float *lh = reinterpret_cast<float *>(base + lay.lh);      // merge: per-head weight sum
    int *misc = reinterpret_cast<int *>(base + lay.misc);      // [0] abort, [1] merge flag, [2] scan carry
    int *scan_tmp = misc + 4;                                  // W+1 warp sums
    const uint32_t ring_addr = base_addr + lay.ring;
    const uint32_t q_addr = base_addr + lay.q;
    const __nv_bfloat16 *q_smem = reinterpret_cast<const __nv_bfloat16 *>(base + lay.q);

    // ---- tiles per sequence, scanned: prefix[b] = tiles of sequences before b ----
    const int Lmax = p.max_pages * p.P;
    if (threadIdx.x == 0) {
        misc[0] = 0;
        misc[2] = 0;
        prefix[0] = 0;
    }
    __syncthreads();
    for (int b0 = 0; b0 < p.B; b0 += NTHR) {
        const int b = b0 + threadIdx.x;
        int n = 0;
        if (b < p.B) {
            int L = p.seq_lens[b];
            if (L < 0 || L > Lmax) {  // an invalid length makes the sequence empty
                if (blockIdx.x == 0) record_status(p.status, PKV_ERR_BAD_SEQ_LEN);
                L = 0;
            }
            n = (L + T - 1) / T;
        }
        int x = n;  // inclusive scan within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scan_tmp[warp] = x;
        __syncthreads();
        int before = misc[2];
        for (int w = 0; w < warp; ++w) before += scan_tmp[w];
        if (b < p.B) prefix[b + 1] = before + x;
        __syncthreads();
        if (threadIdx.x == NTHR - 1) misc[2] = before + x;
        __syncthreads();
    }
    // empty sequences: out = 0 and lse = -inf, spread over the blocks
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (prefix[b + 1] != prefix[b]) continue;
        for (int i = threadIdx.x; i < p.Hq * D / 2; i += NTHR)
            *reinterpret_cast<uint32_t *>(p.out + (size_t)b * p.Hq * D + 2 * i) = 0u;
        if (p.lse)
            for (int i = threadIdx.x; i < p.Hq; i += NTHR) p.lse[(size_t)b * p.Hq + i] = ninf;
    }
    // this block's slice of the tile list.  The list is ordered (kv head, sequence, tile),
    // so blocks whose slices sit one head apart stream the same pages at the same time:
    // the kv heads of a token share DRAM rows, and reading them together keeps rows open.
    const int per_head = prefix[p.B];
    const int total = p.Hkv * per_head;
    const int per = max((total + (int)gridDim.x - 1) / (int)gridDim.x, p.min_range_tiles);
    const int beg = (int)blockIdx.x * per;
    const int end = min(beg + per, total);
    if (beg >= end) return;  // uniform: nothing for this block

    if (threadIdx.x == 0) {
        for (int i = 0; i < W * R; ++i) mbar_init(smem_addr(&full[i]), 1);
        for (int i = 0; i < QS; ++i) {
            mbar_init(smem_addr(&item_full[i]), 1);
            mbar_init(smem_addr(&item_empty[i]), W);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const Waiter waiter{reinterpret_cast<volatile int *>(&misc[0]), p.status, p.wait_limit_ns};

    if (warp == W) {
        // =========================== item warp ===========================
        if (lane == 0) {
            prefetch_tensor_map(&tmK);
            prefetch_tensor_map(&tmV);
        }
        int it = 0;  // items prepared by this block
        int f0 = beg;
        while (f0 < end) {
            // the segment (b, kv head) holding tile f0; the list runs kv head by kv head, and
            // within one head b is the last sequence starting at or before the tile
            const int kvh = f0 / per_head;
            const int r = f0 - kvh * per_head;
            int lo = 0, hi = p.B - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (prefix[mid] <= r) lo = mid; else hi = mid - 1;
            }
            const int b = lo;
            const int nb = prefix[b + 1] - prefix[b];
            const int seg_start = kvh * per_head + prefix[b];
            const int seg_end = seg_start + nb;
            const int pe = min(seg_end, end);
            const bool whole = seg_start >= beg && seg_end <= end;
            int L = p.seq_lens[b];
            if (L < 0 || L > Lmax) L = 0;
            const int mf = seg_start / per;
            const int n_pieces = whole ? 1 : (seg_end - 1) / per - mf + 1;
            const int my_slot = 2 * (int)blockIdx.x + (f0 > beg ? 1 : 0);
            const int mf_tail = seg_start > mf * per ? 1 : 0;
            for (int ta = f0 - seg_start; ta < pe - seg_start; ta += p.max_item_tiles) {
                const int tb = min(ta + p.max_item_tiles, pe - seg_start);
                const int qslot = it % QS;
                waiter.wait(smem_addr(&item_empty[qslot]), ((it / QS) & 1) ^ 1);  // slot released
                const int tok_begin = ta * T;
                const int tok_end = min(tb * T, L);
                const int page_begin = tok_begin >> p.log2P;
                const int npg = ((tok_end - 1) >> p.log2P) + 1 - page_begin;
                // the item's block-table slice; out-of-range ids become -1
                int *slice = tab + qslot * kMaxItemPages;
                int bad = 0;
                for (int i = lane; i < npg; i += 32) {
                    int v = __ldg(p.block_table + (size_t)b * p.max_pages + page_begin + i);
                    if ((unsigned)v >= (unsigned)p.num_pages) {
                        record_status(p.status, PKV_ERR_BAD_PAGE_INDEX);
                        v = -1;
                        bad = 1;
                    }
                    slice[i] = v;
                }
                bad = __any_sync(0xffffffffu, bad);
                __threadfence_block();
                __syncwarp();
                if (lane == 0) {
                    ItemDesc &dsc = desc[qslot];
                    dsc.b = b;
                    dsc.kvh = kvh;
                    dsc.L = L;
                    dsc.tok_begin = tok_begin;
                    dsc.tok_end = tok_end;
                    dsc.page_begin = page_begin;
                    dsc.any_bad = bad;
                    dsc.flags = (ta == f0 - seg_start ? kFirst : 0) | (tb == pe - seg_start ? kLast : 0);
                    dsc.n_pieces = n_pieces;
                    dsc.slot = my_slot;
                    dsc.merge_f = mf;
                    dsc.merge_f_tail = mf_tail;
                    const uint32_t bar = smem_addr(&item_full[qslot]);
                    const uint32_t qbytes = (uint32_t)(G * D * 2);
                    mbar_arrive_expect_tx(bar, qbytes);
                    bulk_copy_g2s(q_addr + (uint32_t)(qslot * H8 * D * 2), p.q + ((size_t)b * p.Hq + kvh * G) * D,
                                  qbytes, bar);
                }
                ++it;
            }
            f0 = pe;
        }
        const int qslot = it % QS;  // end marker
        waiter.wait(smem_addr(&item_empty[qslot]), ((it / QS) & 1) ^ 1);
        if (lane == 0) {
            desc[qslot].flags = kEnd;
            mbar_arrive(smem_addr(&item_full[qslot]));
        }
    } else {
        // =========================== consumer warps ===========================
        const int g = lane >> 2, cc = lane & 3;
        const uint64_t policy = l2_policy_evict_first();
        // Issue cursor: the next of this warp's stages to copy (item ii, stage si), gi copies so far.
        int ii = 0, si = 0, ni = 0, gi = 0;
        bool ii_ready = false, issue_done = false;
        ItemDesc di{};
        // Consume cursor: item ic, gc stages consumed so far.
        int ic = 0, gc = 0;

        // Keeps R of this warp's stages in flight, walking on into later items (at most
        // QS-1 items ahead of the one being consumed, whose slots are already prepared).
        // Only lane 0 runs it: the issue state lives in lane 0 alone, so a wait that gave
        // up cannot make the warp's lanes diverge.
        auto top_up = [&]() {
            while (!issue_done && gi < gc + R) {
                if (!ii_ready) {
                    if (ii > ic + QS - 1) break;
                    waiter.wait(smem_addr(&item_full[ii % QS]), (ii / QS) & 1);
                    di = desc[ii % QS];
                    if (di.flags & kEnd) {
                        issue_done = true;
                        break;
                    }
                    ii_ready = true;
                    si = warp;
                    ni = (di.tok_end - di.tok_begin + T - 1) / T;
                }
                if (si >= ni) {
                    ++ii;
                    ii_ready = false;
                    continue;
                }
                {
                    const int slot = warp * R + gi % R;
                    const int t0 = di.tok_begin + si * T;
                    const int *slice = tab + (ii % QS) * kMaxItemPages;
                    int pages[4];
                    uint32_t bytes = 0;
                    for (int j = 0; j < nbox; ++j) {
                        const int t = t0 + j * box_t;
                        pages[j] = t < di.tok_end ? slice[(t >> p.log2P) - di.page_begin] : -2;
                        if (pages[j] >= 0) bytes += 2 * DC * box_t * 128;
                    }
                    const uint32_t bar = smem_addr(&full[slot]);
                    const uint32_t kdst = ring_addr + (uint32_t)(slot * STAGE);
                    mbar_arrive_expect_tx(bar, bytes);
                    for (int j = 0; j < nbox; ++j) {
                        if (pages[j] < 0) continue;
                        const int row = pages[j] * p.P + ((t0 + j * box_t) & (p.P - 1));
                        if (p.box4 && nbox == 1) {
                            // one box: (64 dims, box_t rows, all D/64 column blocks) per tensor
                            tma_load_4d(kdst, &tmK, 0, row, 0, di.kvh, bar, policy);
                            tma_load_4d(kdst + TILE, &tmV, 0, row, 0, di.kvh, bar, policy);
                        } else {
#pragma unroll
                            for (int dc = 0; dc < DC; ++dc) {
                                const uint32_t off = (uint32_t)(dc * SUB + j * box_t * 128);
                                tma_load_3d(kdst + off, &tmK, dc * 64, di.kvh, row, bar, policy);
                                tma_load_3d(kdst + TILE + off, &tmV, dc * 64, di.kvh, row, bar, policy);
                            }
                        }
                    }
                }
                si += W;
                ++gi;
            }
        };

        // online-softmax state of the current piece
        float acc[KS][NT][4];
        float m_run[NT][2], l_run[NT][2], lt_run[NT][2];

        while (true) {
            if (lane == 0) top_up();
            __syncwarp();
            const int qslot = ic % QS;
            waiter.wait(smem_addr(&item_full[qslot]), (ic / QS) & 1);
            // One thread copies the descriptor between two consumer barriers, so every
            // consumer warp follows the same path (and meets the same barriers) even if
            // a bounded wait gave up.
            consumer_sync(CT);
            if (threadIdx.x == 0) desc[QS] = desc[qslot];
            consumer_sync(CT);
            const ItemDesc d = desc[QS];
            if (d.flags & kEnd) break;
            const size_t row0 = (size_t)d.b * p.Hq + d.kvh * G;

            // query fragments (B operand of the score mma): q^T[d, head]
            uint32_t qf[KS][NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int head = nt * 8 + g;
                const uint32_t *qp =
                    reinterpret_cast<const uint32_t *>(q_smem + (size_t)(qslot * H8 + head) * D + 2 * cc);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qf[ks][nt][0] = head < G ? qp[ks * 8] : 0u;
                    qf[ks][nt][1] = head < G ? qp[ks * 8 + 4] : 0u;
                }
            }
            const int *slice = tab + qslot * kMaxItemPages;
            if (d.flags & kFirst) {
#pragma unroll
                for (int i = 0; i < KS; ++i)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[i][nt][e] = 0.f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        m_run[nt][h2] = ninf;
                        l_run[nt][h2] = 0.f;
                        lt_run[nt][h2] = 0.f;
                    }
            }
            // a key is used if it lies before the item's end and its page id was in range
            auto key_valid = [&](int t) -> bool {
                return t < d.tok_end && slice[(t >> p.log2P) - d.page_begin] >= 0;
            };

            const int n_stages = (d.tok_end - d.tok_begin + T - 1) / T;
            for (int s = warp; s < n_stages; s += W) {
                if (lane == 0) top_up();
                __syncwarp();
                const int slot = warp * R + gc % R;
                waiter.wait(smem_addr(&full[slot]), (gc / R) & 1);
                const int t0 = d.tok_begin + s * T;
                const uint32_t kbase = ring_addr + (uint32_t)(slot * STAGE);
                const uint32_t vbase = kbase + TILE;
                const bool masked = (t0 + T > d.tok_end) || d.any_bad;

                // S^T = K q^T
                float sc[MT][NT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                        const int chunk = (ks & 3) * 2 + (lane >> 4);
                        const uint32_t addr =
                            kbase + (uint32_t)((ks >> 2) * SUB + row * 128 + ((chunk ^ (row & 7)) << 4));
                        uint32_t a0, a1, a2, a3;
                        ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16_16816(sc[mt][nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
                    }
                }

                // scale to log2 units, mask, running max
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float v = sc[mt][nt][e] * p.scale_log2;
                            if (masked && !key_valid(t0 + mt * 16 + g + ((e >> 1) << 3))) v = ninf;
                            sc[mt][nt][e] = v;
                        }
                float alpha[NT][2], mref[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        float mx = ninf;
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) mx = fmaxf(mx, fmaxf(sc[mt][nt][h2], sc[mt][nt][h2 + 2]));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        const float m_new = fmaxf(m_run[nt][h2], mx);
                        const float r = (m_new == ninf) ? 0.f : m_new;
                        alpha[nt][h2] = ex2(m_run[nt][h2] - r);
                        mref[nt][h2] = r;
                        m_run[nt][h2] = m_new;
                        l_run[nt][h2] *= alpha[nt][h2];
                        lt_run[nt][h2] *= alpha[nt][h2];
                    }
#pragma unroll
                for (int i = 0; i < KS; ++i)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        acc[i][nt][0] *= alpha[nt][0];
                        acc[i][nt][1] *= alpha[nt][1];
                        acc[i][nt][2] *= alpha[nt][0];
                        acc[i][nt][3] *= alpha[nt][1];
                    }

                // O^T += V^T P^T, one 16-key tile at a time
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t pb[NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float p0 = ex2(sc[mt][nt][0] - mref[nt][0]), p1 = ex2(sc[mt][nt][1] - mref[nt][1]);
                        const float p2 = ex2(sc[mt][nt][2] - mref[nt][0]), p3 = ex2(sc[mt][nt][3] - mref[nt][1]);
                        const uint32_t x0 = pack_bf16x2(p0, p1);
                        const uint32_t x1 = pack_bf16x2(p2, p3);
                        l_run[nt][0] += p0 + p2;
                        l_run[nt][1] += p1 + p3;
                        lt_run[nt][0] += bf16_lo(x0) + bf16_lo(x1);
                        lt_run[nt][1] += bf16_hi(x0) + bf16_hi(x1);
                        pb[nt][0] = movmatrix_trans(x0);
                        pb[nt][1] = movmatrix_trans(x1);
                    }
                    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
                    if (masked) {
                        const int t = t0 + mt * 16 + 2 * cc;
                        vm0 = (key_valid(t) ? 0x0000ffffu : 0u) | (key_valid(t + 1) ? 0xffff0000u : 0u);
                        vm1 = (key_valid(t + 8) ? 0x0000ffffu : 0u) | (key_valid(t + 9) ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int md = 0; md < KS; ++md) {
                        const int row = mt * 16 + (lane & 7) + (lane >> 4) * 8;
                        const int chunk = (md & 3) * 2 + ((lane >> 3) & 1);
                        const uint32_t addr =
                            vbase + (uint32_t)((md >> 2) * SUB + row * 128 + ((chunk ^ (row & 7)) << 4));
                        uint32_t a0, a1, a2, a3;
                        ldmatrix_x4_trans(addr, a0, a1, a2, a3);
                        a0 &= vm0;
                        a1 &= vm0;
                        a2 &= vm1;
                        a3 &= vm1;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16_16816(acc[md][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    }
                }
                __syncwarp();  // every lane is done with the slot: it may be refilled
                ++gc;
            }
            // the item's slot (query rows, table slice) is no longer needed
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&item_empty[qslot]));
            ++ic;
            if (!(d.flags & kLast)) continue;

            // ---- per-warp finalisation: reduce the denominators over the key rows ----
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    float l = l_run[nt][h2], lt = lt_run[nt][h2];
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        l += __shfl_xor_sync(0xffffffffu, l, o);
                        lt += __shfl_xor_sync(0xffffffffu, lt, o);
                    }
                    l_run[nt][h2] = l;
                    lt_run[nt][h2] = lt;
                }

            // ---- block combine: warps merge pairwise through shared memory into warp 0 ----
            // Every lane holds the same fragment positions in every warp, so the merge is
            // element by element: rescale both sides to the larger running max and add.
            constexpr int NACC = KS * NT * 4;
#pragma unroll
            for (int half = W / 2; half >= 1; half >>= 1) {
                if (warp >= half && warp < 2 * half) {
                    float *sl = red + (warp - half) * TL::SLOT_FLOATS + lane;
                    int k = 0;
#pragma unroll
                    for (int md = 0; md < KS; ++md)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) sl[32 * k++] = acc[md][nt][e];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            sl[32 * k++] = m_run[nt][h2];
                            sl[32 * k++] = l_run[nt][h2];
                            sl[32 * k++] = lt_run[nt][h2];
                        }
                }
                consumer_sync(CT);
                if (warp < half) {
                    const float *sl = red + warp * TL::SLOT_FLOATS + lane;
                    float ra[NT][2], rb[NT][2];
                    int k = NACC;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const float mb = sl[32 * k], lb = sl[32 * (k + 1)], ltb = sl[32 * (k + 2)];
                            k += 3;
                            const float mn = fmaxf(m_run[nt][h2], mb);
                            const float ref = mn == ninf ? 0.f : mn;
                            ra[nt][h2] = ex2(m_run[nt][h2] - ref);
                            rb[nt][h2] = ex2(mb - ref);
                            l_run[nt][h2] = l_run[nt][h2] * ra[nt][h2] + lb * rb[nt][h2];
                            lt_run[nt][h2] = lt_run[nt][h2] * ra[nt][h2] + ltb * rb[nt][h2];
                            m_run[nt][h2] = mn;
                        }
                    k = 0;
#pragma unroll
                    for (int md = 0; md < KS; ++md)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                acc[md][nt][e] = acc[md][nt][e] * ra[nt][e & 1] + sl[32 * k] * rb[nt][e & 1];
                                ++k;
                            }
                }
                consumer_sync(CT);
            }

            // ---- warp 0 writes the piece's result from its registers ----
            const bool whole = d.n_pieces == 1;
            if (warp == 0) {
                float inv[NT][2], lse_v[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const bool empty_col = m_run[nt][h2] == ninf;
                        inv[nt][h2] = empty_col ? 0.f : 1.f / lt_run[nt][h2];
                        lse_v[nt][h2] = empty_col ? ninf : (m_run[nt][h2] + __log2f(l_run[nt][h2])) * kLn2;
                    }
                if (whole) {  // the whole segment: final bf16 output and lse
#pragma unroll
                    for (int md = 0; md < KS; ++md)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int head = nt * 8 + 2 * cc + (e & 1);
                                const int dd = md * 16 + g + ((e >> 1) << 3);
                                if (head < G)
                                    p.out[(row0 + head) * D + dd] = __float2bfloat16_rn(acc[md][nt][e] * inv[nt][e & 1]);
                            }
                    if (g == 0 && p.lse)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int head = nt * 8 + 2 * cc + h2;
                                if (head < G) p.lse[row0 + head] = lse_v[nt][h2];
                            }
                } else {  // a piece of the segment: normalised output and lse into this block's slot
                    float *po = p.part_out + (size_t)d.slot * G * D;
#pragma unroll
                    for (int md = 0; md < KS; ++md)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int head = nt * 8 + 2 * cc + (e & 1);
                                const int dd = md * 16 + g + ((e >> 1) << 3);
                                if (head < G) po[(size_t)head * D + dd] = acc[md][nt][e] * inv[nt][e & 1];
                            }
                    if (g == 0)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const int head = nt * 8 + 2 * cc + h2;
                                if (head < G) p.part_lse[(size_t)d.slot * G + head] = lse_v[nt][h2];
                            }
                    __threadfence();
                }
            }
            if (!whole) {
                // the block that finishes the segment's last piece merges all of them;
                // atomicInc wraps the segment's counter back to 0 for the next call
                consumer_sync(CT);
                if (threadIdx.x == 0)
                    misc[1] = atomicInc(reinterpret_cast<unsigned *>(p.counters + d.b * p.Hkv + d.kvh),
                                        (unsigned)(d.n_pieces - 1)) == (unsigned)(d.n_pieces - 1);
                consumer_sync(CT);
                if (misc[1]) {
                    __threadfence();
                    merge_pieces<D, W>(p, d, row0, mh, lh, lane, warp);
                }
            }
            consumer_sync(CT);  // the combine buffer and merge scratch may be reused
        }
    }
}

// Bounded-wait self-test: waits on a barrier nothing completes.
__global__ void wait_timeout_selftest_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(smem_addr(&bar), 0, limit_ns)) record_status(status, PKV_ERR_DEVICE_TIMEOUT);
}

}  // namespace pkv
