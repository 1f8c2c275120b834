// plan.h -- the host planner: split count, tiling and workspace layout as a
// pure function of (shape, SM count).  No CUDA calls.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pkv.h"

namespace pkv {

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__ __forceinline__
#else
#define PKV_HD inline
#endif

// Compile-time tiling of one decode-kernel variant, chosen by head dim D.
//   T: keys per pipeline stage (a multiple of the 16-row mma tile)
//   W: consumer warps per block, each streaming its own stages
template <int D>
struct Tiling;
template <>
struct Tiling<64> { static constexpr int T = 32, W = 4; };
template <>
struct Tiling<128> { static constexpr int T = 16, W = 4; };
template <>
struct Tiling<256> { static constexpr int T = 16, W = 4; };

struct RuntimeTiling {
    int T, W;
};
RuntimeTiling tiling_for(int D);

// Number of 8-wide head tiles (mma N tiles) for group size G.
inline int head_tiles(int G) { return G <= 8 ? 1 : (G <= 16 ? 2 : 4); }

// Fewest keys a split takes (the plan's rule, and the device's adaptive chunk).
constexpr int kMinSplitTokens = 256;

// The block slots the one-wave split rule counts: every resident block for the fp8 cache, at
// most two per SM for a bf16 cache (fewer, longer splits amortise a block's start-up better).
PKV_HD int split_slots(int num_sms, int blocks_per_sm, bool kv8)
{
    return num_sms * (kv8 ? blocks_per_sm : (blocks_per_sm < 2 ? blocks_per_sm : 2));
}

// Most (token, head) rows one decode block serves: 32, or 16 at D = 256, where the 32-row
// variant's accumulators and query fragments exceed the register file and spill (measured:
// ~2.6 KB of spills a thread, 9x slower than two 16-row blocks).
PKV_HD constexpr int max_block_rows(int D) { return D == 256 ? 16 : 32; }

// Most splits whose partials merge inside a thread-block cluster (the portable cluster size).
constexpr int kMaxClusterSplits = 8;

// Resident blocks per SM a variant is compiled for (its launch bound, so its register
// budget).  Variants with one head tile are light enough for three, which hides more
// latency; D = 256 bf16 tiles fill shared memory with one block, fp8 ones with two.
PKV_HD constexpr int target_blocks(int D, int NT, bool kv8)
{
    return D == 256 ? ((kv8 && NT <= 2) ? 2 : 1) : NT == 1 ? 3 : 2;
}

// Keys per stage: the fp8 kernel with one head tile at D = 128 takes 32 (two mma
// tiles), so the per-stage work (wait, copy issue, scale bookkeeping) is spread over
// twice the keys; everything else takes the tiling's T.
PKV_HD constexpr int stage_keys(int D, int NT, bool kv8) { return (kv8 && D == 128 && NT == 1) ? 32 : (D == 64 ? 32 : 16); }

// Ring depth per warp (stages in flight), sized so a block's ring fits its share of
// shared memory: an fp8 stage is half the bytes of a bf16 one.
PKV_HD constexpr int ring_depth(int D, int NT, bool kv8)
{
    return D == 256 ? (kv8 ? (target_blocks(D, NT, kv8) == 2 ? 3 : 6) : 3)
                    : target_blocks(D, NT, kv8) >= 3 ? (kv8 ? (stage_keys(D, NT, kv8) == 32 && D == 128 ? 2 : 4) : 2)
                                                     : (kv8 ? 6 : 3);
}

// Shared-memory carve-up of one decode block (byte offsets from a 1024-aligned
// base).  The kernel and the planner both use this, so they cannot disagree.
struct SmemLayout {
    int ring;      // W*R stages of [K tile | V tile]; bf16: T x D bf16 per tile, 128B-swizzled;
                   // fp8: T x D e4m3 codes per tile, 128B-swizzled (64B for D = 64)
    int scales;    // fp8 only: W*R stages of [K scales | V scales], T f32 each
    int bars;      // W*R mbarriers (8 B each)
    int m;         // [W][H8] f32 running max per warp (log2 units)
    int l;         // [W][H8] f32 softmax denominator per warp (sum of the f32 probabilities)
    int lt;        // [W][H8] f32 same, summed over the bf16-rounded probabilities the PV mma uses
    int f;         // [W][H8] f32 per-warp combine factor
    int lse;       // [H8] f32 block result per head
    int flag;      // one int: "this block merges its group"
    int xbar;      // cluster merge: two mbarriers (8 B each): "ready" (split 0's ring is free for
                   // the partials), "full" (every partial has landed in split 0's ring)
    int recv;      // cluster merge, split 0 only: the partials of splits 1 .. S-1, `recv_slot`
    int recv_slot; // bytes apart, in the ring after the combine buffer: [H8][D] f32 outputs then
                   // [H8] f32 lse each
    int table;     // block_table slice (int32), `table_entries` of them
    int table_entries;
    int total;     // bytes from the aligned base
    int dynamic;   // bytes to request (total + alignment slack)
};

PKV_HD int round_up_int(int x, int m) { return (x + m - 1) / m * m; }

// Bytes of one ring stage (K and V tiles; a multiple of 1024 for every tiling).
PKV_HD int stage_bytes(int D, int T, bool kv8) { return kv8 ? 2 * T * D : 2 * T * D * 2; }

PKV_HD SmemLayout smem_layout(int D, int T, int W, int R, int NT, int chunk_tokens, int page_size,
                              bool kv8 = false)
{
    SmemLayout s;
    const int H8 = NT * 8;
    const int ring = W * R * stage_bytes(D, T, kv8);
    const int scales = kv8 ? W * R * 2 * T * 4 : 0;
    const int red = W * H8 * (D + 4) * 4;  // per-warp f32 accumulators, reuses the ring
    s.ring = 0;
    s.scales = ring;
    s.bars = round_up_int(ring + scales > red ? ring + scales : red, 1024);
    s.m = s.bars + W * R * 8;
    s.l = s.m + W * H8 * 4;
    s.lt = s.l + W * H8 * 4;
    s.f = s.lt + W * H8 * 4;
    s.lse = s.f + W * H8 * 4;
    s.flag = s.lse + H8 * 4;
    s.xbar = round_up_int(s.flag + 4, 8);
    s.recv = round_up_int(red, 128);
    s.recv_slot = round_up_int(H8 * (D + 1) * 4, 128);
    s.table = round_up_int(s.xbar + 16, 16);
    s.table_entries = chunk_tokens / page_size + 2;
    s.total = round_up_int(s.table + s.table_entries * 4, 16);
    s.dynamic = s.total + 1024;
    return s;
}

// Whether a decode launch of S splits can merge them inside a cluster: 2 <= S <= 8 and split
// 0's ring holds the combine buffer and the other splits' partials.
PKV_HD bool cluster_merge_fits(const SmemLayout &lay, int S, int ring_bytes)
{
    return S >= 2 && S <= kMaxClusterSplits && lay.recv + (S - 1) * lay.recv_slot <= ring_bytes;
}

// Workspace layout (byte offsets), used only when S > 1:
//   [0, 256)   header: int32 status word at 0
//   counters   B*Hkv int32 split-completion counters (zero before first use; self-resetting)
//   part_lse   S*B*Hq f32
//   part_out   S*B*Hq*D f32
// With S == 1 the workspace is the 256-byte header alone.
constexpr size_t kWorkspaceHeader = 256;
struct WorkspaceLayout {
    size_t counters, part_lse, part_out, total;
};
// n_counters: one per (sequence, kv head, query tile); total_rows: rows of out (B*Hq for decode).
WorkspaceLayout workspace_layout(int S, size_t n_counters, size_t total_rows, int D);

// Shape checks shared by every entry point (no CUDA call).
pkv_status validate_shape(int B, int Hq, int Hkv, int D, int page_size, int max_pages);

// Validates the shape (not pointers) and fills `plan` for the bf16-cache kernel or,
// with kv8, the fp8-cache one.  group_rows: (token, query head) rows of one (sequence,
// kv head) group, at most max_q_len * G (0: decode, G rows); total_rows: rows of the
// output, total_q * Hq (0: B * Hq).
// allow_cluster: a decode plan with 2-8 splits may merge them inside a thread-block cluster
// (plan->merge_needed = 2) when split 0's ring holds the partials.
pkv_status make_plan(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                     int num_splits, pkv_plan *plan, bool kv8 = false, long group_rows = 0, long total_rows = 0,
                     bool allow_cluster = false);

}  // namespace pkv
