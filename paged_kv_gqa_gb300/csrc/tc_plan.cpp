// tc_plan.cpp -- key splits of the tensor-core several-rows kernels (a pure host function
// of the shape and the SM count, like the decode planner).
#include "tc_plan.h"

#include <algorithm>

namespace pkv {

TcSplit tc_split_plan(int B, int Hq, int Hkv, int page_size, int max_pages, int total_q, int max_q_len,
                      int num_splits, int cta_rows, int num_sms)
{
    TcSplit t;
    const long G = Hkv > 0 ? Hq / Hkv : 1;
    const long max_tiles = std::max(1l, ((long)max_pages * page_size + 127) / 128);
    t.q_tiles = (int)(((long)max_q_len * G + cta_rows - 1) / cta_rows);
    const long groups = std::max(1l, (long)B * Hkv * t.q_tiles);
    long S;
    if (num_splits > 0)
        S = num_splits;
    else if (groups < num_sms)
        S = num_sms / groups;
    else
        S = (max_tiles + kTcChunkTiles - 1) / kTcChunkTiles;
    S = std::min(std::max(S, 1l), std::min(max_tiles, 65535l));
    const long chunk = (max_tiles + S - 1) / S;
    t.chunk_tiles = (int)chunk;
    t.splits = (int)((max_tiles + chunk - 1) / chunk);
    t.ws = workspace_layout(t.splits, (size_t)B * t.q_tiles * Hkv, (size_t)total_q * Hq, 128);
    return t;
}

}  // namespace pkv
