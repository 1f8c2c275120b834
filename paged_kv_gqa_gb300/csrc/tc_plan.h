// tc_plan.h -- host planner of the tensor-core several-rows kernels' key splits.
#pragma once

#include "plan.h"

namespace pkv {

// Key splits of the tensor-core several-rows kernels (prefill_tc_kernel.cuh with 128 rows
// per CTA, prefill_tc2_kernel.cuh with 256, prefill_tc256_kernel.cuh at D = 256): a CTA takes
// chunk_tiles key tiles (tc_tile_keys(D) keys each) of its group.  num_splits > 0: that many chunks over the table width.  num_splits = 0: with
// fewer (sequence, kv head, query tile) groups than SMs, the count S (at most 4 * num_sms /
// groups) that minimises ceil(groups * S / num_sms) * (ceil(tiles / S) + the CTA cost in tiles),
// the CTA waves times each CTA's tiles plus its fixed cost (Q load, first copies, epilogue,
// merge; measured on GB300 as about 2048 keys' time); otherwise chunks of at most
// kTcChunkKeys keys, which only the longest groups of a ragged batch exceed.
// The workspace holds the per-split partials and one counter per group when splits > 1.
// Tiles of 128 keys at D = 128, of 64 keys at D = 256 (prefill_tc256_kernel.cuh); the chunk
// cap (8192 keys) and the CTA cost (2048 keys' time) are the same in keys either way.
constexpr int kTcChunkKeys = 8192;
constexpr long kTcCtaCostKeys = 2048;
struct TcSplit {
    int splits, chunk_tiles, q_tiles;
    WorkspaceLayout ws;
};
TcSplit tc_split_plan(int B, int Hq, int Hkv, int page_size, int max_pages, int total_q, int max_q_len,
                      int num_splits, int cta_rows, int num_sms, int D = 128);
inline int tc_tile_keys(int D) { return D == 256 ? 64 : 128; }

}  // namespace pkv
