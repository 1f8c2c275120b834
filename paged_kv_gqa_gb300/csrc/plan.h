// plan.h -- the host planner: split count, tiling and workspace layout as a
// pure function of (shape, SM count).  No CUDA calls.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pkv.h"

namespace pkv {

#if defined(__CUDACC__)
#define PKV_HDC __host__ __device__
#else
#define PKV_HDC
#endif

// Sequences per launch: each block scans the batch's lengths into shared memory.
// Larger batches are cut into several launches on the same stream.
constexpr int kMaxBatchPerLaunch = 1024;
// Block-table entries one work item may span (its chunk plus two partial pages).
constexpr int kMaxItemPages = 256;
constexpr int kSmemPerBlockMax = 232448;  // 227 KiB opt-in maximum per block on sm_100-class parts
constexpr int kDescBytes = 48;            // one work-item descriptor

// Compile-time tiling of the persistent decode kernel for head dim D and NT
// 8-wide head tiles (G <= 8 * NT):
//   T   keys per pipeline stage (one 16-key mma tile, two for D = 64)
//   W   consumer warps (8; 4 when the accumulators or the D = 256 stages need the
//       room; 2 for D = 256 with G > 16); one more warp prepares work items
//   QS  work-item slots (query rows, block-table slice, descriptor)
//   R   stages in flight per consumer warp, as many as the 227 KiB of shared
//       memory allow (2..4); each consumer warp issues its own TMA copies
template <int D, int NT>
struct PTiling {
    static constexpr int T = D == 64 ? 32 : 16;
    static constexpr int W = (D == 256 && NT == 4) ? 2 : ((NT == 4 || D == 256) ? 4 : 8);
    static constexpr int QS = 3;
    static constexpr int H8 = 8 * NT;
    static constexpr int STAGE = 2 * T * D * 2;
    // One warp's online-softmax state (O^T fragments, then m, l, lt per column) in
    // lane-major order: the unit the block combine passes between warps.
    static constexpr int SLOT_FLOATS = (D / 16 * NT * 4 + NT * 2 * 3) * 32;
    static PKV_HDC constexpr int fixed_bytes()
    {
        return QS * H8 * D * 2                  // staged query rows
               + QS * kMaxItemPages * 4         // block-table slices
               + (W / 2) * SLOT_FLOATS * 4      // pairwise-combine buffer
               + 2 * H8 * 4                     // per-head max / weight sum of the merge
               + (kMaxBatchPerLaunch + 1) * 4   // per-sequence item prefix
               + (QS + 1) * kDescBytes + 64 * 4 // descriptors (+ the consumers' copy), misc
               + 2 * QS * 8 + 1024 + 512;       // item barriers, alignment slack, rounding
    }
    static constexpr int R_fit = (kSmemPerBlockMax - fixed_bytes()) / (W * (STAGE + 8));
    static constexpr int R = R_fit > 4 ? 4 : R_fit;
};

PKV_HDC constexpr int round_up_c(int x, int m) { return (x + m - 1) / m * m; }

// Shared-memory carve-up of one block (byte offsets from a 1024-aligned base).
struct PersistLayout {
    int ring, q, tab, red, mh, lh, prefix, desc, full, item_full, item_empty, misc;
    int total;    // bytes from the aligned base
    int dynamic;  // bytes to request (total + alignment slack)
};

template <int D, int NT>
PKV_HDC constexpr PersistLayout persist_layout()
{
    using TL = PTiling<D, NT>;
    PersistLayout s{};
    s.ring = 0;
    s.q = TL::W * TL::R * TL::STAGE;
    s.tab = round_up_c(s.q + TL::QS * TL::H8 * D * 2, 16);
    s.red = s.tab + TL::QS * kMaxItemPages * 4;
    s.mh = s.red + (TL::W / 2) * TL::SLOT_FLOATS * 4;
    s.lh = s.mh + TL::H8 * 4;
    s.prefix = s.lh + TL::H8 * 4;
    s.desc = round_up_c(s.prefix + (kMaxBatchPerLaunch + 1) * 4, 16);
    s.full = round_up_c(s.desc + (TL::QS + 1) * kDescBytes, 8);
    s.item_full = s.full + TL::W * TL::R * 8;
    s.item_empty = s.item_full + TL::QS * 8;
    s.misc = s.item_empty + TL::QS * 8;
    s.total = round_up_c(s.misc + 64 * 4, 16);
    s.dynamic = s.total + 1024;
    return s;
}

// Runtime view of the compile-time tiling of the variant a shape selects.
struct RuntimeTiling {
    int T, W, R, smem;
};
RuntimeTiling tiling_for(int D, int NT);

// Number of 8-wide head tiles (mma N tiles) for group size G.
inline int head_tiles(int G) { return G <= 8 ? 1 : (G <= 16 ? 2 : 4); }

// Workspace layout (byte offsets):
//   [0, 256)   header: int32 status word at 0 (zero before first use)
//   counters   B*Hkv int32 piece-completion counters (zero before first use; the kernel
//              returns each to zero)
//   part_lse   2*grid*G f32   two partial slots per block
//   part_out   2*grid*G*D f32
// Batches above kMaxBatchPerLaunch reuse one workspace sized for kMaxBatchPerLaunch sequences.
constexpr size_t kWorkspaceHeader = 256;
struct WorkspaceLayout {
    size_t counters, part_lse, part_out, total;
};
WorkspaceLayout workspace_layout(int grid, int B, int Hq, int Hkv, int D);

// Shape checks shared by every entry point (no CUDA call).
pkv_status validate_shape(int B, int Hq, int Hkv, int D, int page_size, int max_pages);

// Validates the shape (not pointers) and fills `plan`.
pkv_status make_plan(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                     int num_splits, pkv_plan *plan);

}  // namespace pkv
