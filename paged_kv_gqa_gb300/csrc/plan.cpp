// plan.cpp -- host planner for the split-KV decode launch.
//
// The split count is a pure function of the shape and the SM count (OASR
// "Kernel Layer", "Fused attention": never of capture state, because it sets
// the order the f32 partials are summed).  The device-side lengths are not
// visible here, so the plan sizes splits for sequences of full table width.
// The rule (tuned on GB300 by sweeping the split count per workload):
//   - about one wave of blocks: enough splits that every resident block slot
//     gets one, since fewer, larger blocks amortise each block's start-up and
//     epilogue; a batch that already fills the slots is not split;
//   - a split holds at most ~2 MiB of cache bytes (kMaxSplitBytes: K and V, and
//     for the fp8 cache their scales), so that no split becomes a straggler;
//     where this bound sets the count and the blocks span more than one wave,
//     the count in [S, 1.5 S] that fills the last wave of resident blocks best;
//   - never fewer than kMinSplitTokens keys per split.
// The fp8-cache kernel has its own footprint and residency, so its own split count.
// Splits that start past a sequence's length exit at once and are ignored by
// the merge (FlashQuant wiki "CUDA Kernels", paged_decode.cu "Early Exit for
// Empty Splits").
#include "plan.h"

#include <algorithm>
#include <cmath>

namespace pkv {

namespace {
constexpr long kMaxSplitBytes = 2l << 20;  // cache bytes of one (b, kv head) split
constexpr int kSmemPerSm = 233472;          // 228 KiB per SM on sm_100-class parts
constexpr int kSmemPerBlockMax = 232448;    // 227 KiB opt-in maximum per block
constexpr int kBlockReserve = 1024;         // shared memory the system reserves per block
constexpr int kMaxTablePages = 4096;        // block_table slice a block stages in smem
}  // namespace

RuntimeTiling tiling_for(int D)
{
    switch (D) {
        case 64: return {Tiling<64>::T, Tiling<64>::W};
        case 128: return {Tiling<128>::T, Tiling<128>::W};
        case 256: return {Tiling<256>::T, Tiling<256>::W};
        default: return {0, 0};
    }
}

static size_t pad256(size_t x) { return (x + 255) / 256 * 256; }

WorkspaceLayout workspace_layout(int S, size_t n_counters, size_t total_rows, int D)
{
    WorkspaceLayout w;
    w.counters = kWorkspaceHeader;
    w.part_lse = w.counters + pad256(n_counters * sizeof(int));
    w.part_out = w.part_lse + pad256((size_t)S * total_rows * sizeof(float));
    w.total = S <= 1 ? kWorkspaceHeader : w.part_out + (size_t)S * total_rows * D * sizeof(float);
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
                     int num_splits, pkv_plan *plan, bool kv8, long group_rows, long total_rows,
                     bool allow_cluster)
{
    if (!plan || num_sms <= 0 || num_splits < 0 || group_rows < 0 || total_rows < 0) return PKV_ERR_INVALID_ARG;
    const pkv_status v = validate_shape(B, Hq, Hkv, D, page_size, max_pages);
    if (v != PKV_OK) return v;
    const int G = Hq / Hkv;

    // A block serves up to 32 (token, query head) rows of one (sequence, kv head) group
    // (all G heads of a decode step), 16 at D = 256 (32 rows there need more registers
    // than a thread has and spill); longer groups take several query tiles.
    const long rows = group_rows > 0 ? group_rows : G;
    const int NT = head_tiles((int)std::min<long>(rows, max_block_rows(D)));
    const long q_tiles = (rows + NT * 8 - 1) / (NT * 8);
    if ((long)B * Hkv * q_tiles >= (1l << 31)) return PKV_ERR_INVALID_ARG;
    if (B > 65535) return PKV_ERR_UNSUPPORTED;  // sequences are the grid's z dimension
    const long out_rows = total_rows > 0 ? total_rows : (long)B * Hq;

    RuntimeTiling t = tiling_for(D);
    t.T = stage_keys(D, NT, kv8);
    const int max_tokens = max_pages * page_size;
    const int units = std::max(1, (int)(B * Hkv * q_tiles));

    // Resident blocks per SM: the shared-memory limit (sized with the largest table slice
    // the auto plan uses) or the variant's register budget, whichever is lower.
    const int R = ring_depth(D, NT, kv8);
    const long token_bytes = kv8 ? 2l * D + 8 : 4l * D;  // K and V of one token and kv head (+ fp8 scales)
    const int cap_tokens = std::max(t.T, (int)(kMaxSplitBytes / token_bytes) / t.T * t.T);
    const SmemLayout ref = smem_layout(D, t.T, t.W, R, NT, cap_tokens, page_size, kv8);
    int per_sm = std::max(1, kSmemPerSm / (ref.dynamic + kBlockReserve));
    per_sm = std::min(per_sm, target_blocks(D, NT, kv8));
    // The split rule counts at most two slots per SM for a bf16 cache: its blocks carry
    // twice the bytes per key, and fewer, longer splits amortise their start-up better
    // (measured on GB300: the batch workload runs fastest at 4-5 splits with three
    // blocks resident, at 8 with the fp8 cache).
    const int slots = split_slots(num_sms, per_sm, kv8);

    const int max_stage_splits = (max_tokens + t.T - 1) / t.T;
    int S;
    if (num_splits > 0) {
        S = std::min(num_splits, max_stage_splits);
    } else {
        // About one wave of blocks: enough splits that every resident slot gets one, but no
        // more blocks than are resident at once (a second, nearly empty wave costs a whole
        // block's time).  Fewer (larger) blocks amortise each block's fixed start-up and
        // epilogue cost; a batch that already has a block per slot is not split at all.
        S = std::max(1, (slots + units - 1) / units);
        if ((long)units * S > (long)num_sms * per_sm) S = std::max(1, num_sms * per_sm / units);
        // Bound the bytes of one split so that no split becomes a straggler.  Where that
        // bound sets the count and the blocks span more than one wave of resident blocks,
        // take the count in [S, 1.5 S] that fills the last wave best (measured on GB300:
        // the long-context workload runs 12% faster (fp8) and 2% faster (bf16) at these
        // counts than with splits of half the size, whose start-up, epilogue and merge
        // cost more than the finer grain gains).
        const int s_cap = (max_tokens + cap_tokens - 1) / cap_tokens;
        if (s_cap > S) {
            S = s_cap;
            const int resident = num_sms * per_sm;
            if ((long)units * S > resident) {
                const int s_lo = S, s_hi = S + S / 2;
                double best = -1.0;
                for (int s = s_lo; s <= s_hi; ++s) {
                    const double waves = (double)units * s / resident;
                    const double eff = waves / std::ceil(waves);
                    if (eff > best + 0.005) {
                        best = eff;
                        S = s;
                    }
                }
            }
        }
        // Never thinner than kMinSplitTokens keys per split.
        S = std::min(S, std::max(1, max_tokens / kMinSplitTokens));
    }
    S = std::max(1, S);
    int chunk = (max_tokens + S - 1) / S;
    chunk = (chunk + t.T - 1) / t.T * t.T;
    // A block stages its block_table slice in shared memory: bound it.
    const int max_chunk = (kMaxTablePages - 2) * page_size;
    if (chunk > max_chunk) chunk = max_chunk / t.T * t.T;
    S = (max_tokens + chunk - 1) / chunk;
    if ((long)S * Hkv * q_tiles * B >= (1l << 31)) return PKV_ERR_INVALID_ARG;

    const SmemLayout lay = smem_layout(D, t.T, t.W, R, NT, chunk, page_size, kv8);
    if (lay.dynamic > kSmemPerBlockMax) return PKV_ERR_UNSUPPORTED;
    per_sm = std::max(1, std::min(kSmemPerSm / (lay.dynamic + kBlockReserve), target_blocks(D, NT, kv8)));

    plan->num_splits = S;
    plan->chunk_tokens = chunk;
    plan->stage_tokens = t.T;
    plan->warps = t.W;
    plan->ring_stages = R;
    plan->blocks_per_sm = per_sm;
    plan->grid_blocks = (int)(S * Hkv * q_tiles * B);
    plan->smem_bytes = lay.dynamic;
    // Decode (one row per sequence, one query tile) with 2-8 splits merges them inside a thread-block cluster
    // through split 0's shared memory; otherwise the last split to finish merges through
    // the workspace.
    // Only grids of one wave (every block resident at once): clusters of S blocks placed whole
    // leave slots idle when blocks of many waves come and go (measured on GB300: the ragged
    // workload's 3584 blocks ran 3-40% slower in clusters of 7-8).
    const bool one_wave = (long)S * Hkv * q_tiles * B <= (long)num_sms * per_sm;
    const bool cluster = allow_cluster && group_rows == 0 && q_tiles == 1 && one_wave &&
                         cluster_merge_fits(lay, S, t.W * R * stage_bytes(D, t.T, kv8));
    plan->merge_needed = S > 1 ? (cluster ? 2 : 1) : 0;
    plan->workspace_bytes = workspace_layout(S, (size_t)B * Hkv * q_tiles, (size_t)out_rows, D).total;
    plan->q_tiles = (int)q_tiles;
    plan->rows_per_block = NT * 8;
    return PKV_OK;
}

}  // namespace pkv
