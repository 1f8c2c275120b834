// tc_plan.h -- host planner of the tensor-core several-rows kernels' key splits.
#pragma once

#include "plan.h"

namespace pkv {

// Key splits of the tensor-core several-rows kernels (prefill_tc_kernel.cuh with 128 rows
// per CTA, prefill_tc2_kernel.cuh with 256): a CTA takes chunk_tiles tiles of 128 keys of
// its group.  num_splits > 0: that many chunks over the table width.  num_splits = 0: with
// fewer (sequence, kv head, query tile) groups than SMs, the count S (at most 4 * num_sms /
// groups) that minimises ceil(groups * S / num_sms) * (ceil(tiles / S) + kTcCtaCostTiles),
// the CTA waves times each CTA's tiles plus its fixed cost (Q load, first copies, epilogue,
// merge; measured on GB300 as about 16 tiles' time); otherwise chunks of at most
// kTcChunkTiles tiles (8192 keys), which only the longest groups of a ragged batch exceed.
// The workspace holds the per-split partials and one counter per group when splits > 1.
constexpr int kTcChunkTiles = 64;
constexpr long kTcCtaCostTiles = 16;
struct TcSplit {
    int splits, chunk_tiles, q_tiles;
    WorkspaceLayout ws;
};
TcSplit tc_split_plan(int B, int Hq, int Hkv, int page_size, int max_pages, int total_q, int max_q_len,
                      int num_splits, int cta_rows, int num_sms);

}  // namespace pkv
