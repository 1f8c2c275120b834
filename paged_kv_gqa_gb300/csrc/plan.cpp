// plan.cpp -- host planner for the balanced persistent decode launch.
//
// The grid is one block per SM.  The device splits the batch's key tiles into
// equal slices, one per block, from seq_lens (a deterministic function of the
// lengths and the SM count; OASR "Kernel Layer", "Fused attention": the split
// must not depend on capture state, since it sets the order the f32 partials
// are summed).  The host only fixes:
//   - the minimum slice (kMinRangeTokens keys, or max_tokens / num_splits when a
//     split count is forced), so that tiny batches are not cut into slivers whose
//     partials cost more than they save;
//   - the largest work item (kMaxItemPages pages of block table staged in shared
//     memory);
//   - the workspace: a header, one counter per (b, kv head), two partial slots per block.
#include "plan.h"

#include <algorithm>
#include <cmath>

namespace pkv {

namespace {
constexpr int kMinRangeTokens = 256;
}  // namespace

template <int D, int NT>
static RuntimeTiling tiling_of()
{
    using TL = PTiling<D, NT>;
    return {TL::T, TL::W, TL::R, persist_layout<D, NT>().dynamic};
}

RuntimeTiling tiling_for(int D, int NT)
{
#define PKV_T(DD, NN) \
    if (D == DD && NT == NN) return tiling_of<DD, NN>();
    PKV_T(64, 1) PKV_T(64, 2) PKV_T(64, 4)
    PKV_T(128, 1) PKV_T(128, 2) PKV_T(128, 4)
    PKV_T(256, 1) PKV_T(256, 2) PKV_T(256, 4)
#undef PKV_T
    return {0, 0, 0, 0};
}

static size_t pad256(size_t x) { return (x + 255) / 256 * 256; }

WorkspaceLayout workspace_layout(int grid, int B, int Hq, int Hkv, int D)
{
    const size_t G = (size_t)(Hq / Hkv);
    WorkspaceLayout w;
    w.counters = kWorkspaceHeader;
    w.part_lse = w.counters + pad256((size_t)B * Hkv * sizeof(int));
    w.part_out = w.part_lse + pad256(2 * (size_t)grid * G * sizeof(float));
    w.total = w.part_out + 2 * (size_t)grid * G * D * sizeof(float);
    return w;
}

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

pkv_status validate_shape(int B, int Hq, int Hkv, int D, int page_size, int max_pages)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || max_pages <= 0) return PKV_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PKV_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return PKV_ERR_UNSUPPORTED;
    if (!is_pow2(page_size) || page_size < 8 || page_size > 256) return PKV_ERR_UNSUPPORTED;
    if ((long)max_pages * page_size >= (1l << 30)) return PKV_ERR_INVALID_ARG;
    if (Hq / Hkv > 32) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

pkv_status make_plan(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_sms,
                     int num_splits, pkv_plan *plan)
{
    if (!plan || num_sms <= 0 || num_splits < 0) return PKV_ERR_INVALID_ARG;
    const pkv_status v = validate_shape(B, Hq, Hkv, D, page_size, max_pages);
    if (v != PKV_OK) return v;
    const int G = Hq / Hkv;
    const int NT = head_tiles(G);
    const RuntimeTiling t = tiling_for(D, NT);
    if (t.smem > kSmemPerBlockMax) return PKV_ERR_UNSUPPORTED;
    const int Bl = std::max(1, std::min(B, kMaxBatchPerLaunch));  // sequences per launch
    const int max_tokens = max_pages * page_size;
    const int max_tiles = (max_tokens + t.T - 1) / t.T;
    const int grid = num_sms;
    if ((long)Bl * Hkv * max_tiles >= (1l << 31)) return PKV_ERR_INVALID_ARG;  // tile indices are int32

    const int min_range = num_splits > 0 ? std::max(1, (max_tiles + num_splits - 1) / num_splits)
                                         : std::max(1, (kMinRangeTokens + t.T - 1) / t.T);
    const int max_item = std::max(1, (kMaxItemPages - 2) * page_size / t.T);
    // Estimates for sequences of full table width (the device uses the real lengths).
    const long total_full = (long)Bl * Hkv * max_tiles;
    const long per_full = std::max((total_full + grid - 1) / grid, (long)min_range);
    const int pieces = (int)std::min<long>((max_tiles + per_full - 1) / per_full + (max_tiles % per_full ? 1 : 0),
                                           grid);

    plan->num_splits = std::max(1, pieces);
    plan->chunk_tokens = min_range * t.T;
    plan->stage_tokens = t.T;
    plan->warps = t.W;
    plan->ring_stages = t.R;
    plan->blocks_per_sm = 1;
    plan->grid_blocks = grid;
    plan->smem_bytes = t.smem;
    plan->merge_needed = pieces > 1 ? 1 : 0;
    plan->max_item_tiles = max_item;
    plan->workspace_bytes = workspace_layout(grid, Bl, Hq, Hkv, D).total;
    return PKV_OK;
}

}  // namespace pkv
