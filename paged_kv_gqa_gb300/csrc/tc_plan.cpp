// tc_plan.cpp -- key splits of the tensor-core several-rows kernels (a pure host function
// of the shape and the SM count, like the decode planner).
#include "tc_plan.h"

#include <algorithm>

namespace pkv {

TcSplit tc_split_plan(int B, int Hq, int Hkv, int page_size, int max_pages, int total_q, int max_q_len,
                      int num_splits, int cta_rows, int num_sms, int D)
{
    TcSplit t;
    const long G = Hkv > 0 ? Hq / Hkv : 1;
    const long tile = tc_tile_keys(D);
    const long max_tiles = std::max(1l, ((long)max_pages * page_size + tile - 1) / tile);
    const long cost_tiles = kTcCtaCostKeys / tile, chunk_tiles = kTcChunkKeys / tile;
    t.q_tiles = (int)(((long)max_q_len * G + cta_rows - 1) / cta_rows);
    const long groups = std::max(1l, (long)B * Hkv * t.q_tiles);
    long S;
    if (num_splits > 0) {
        S = num_splits;
    } else if (groups < num_sms) {
        // a sparse grid: the count whose waves x (tiles per CTA + a CTA's fixed cost) is
        // least, up to four CTAs per SM's worth of splits; ties keep the smaller count
        const long s_max = std::max(1l, std::min(max_tiles, 4l * num_sms / groups));
        long best = -1;
        S = 1;
        for (long s = 1; s <= s_max; ++s) {
            const long waves = (groups * s + num_sms - 1) / num_sms;
            const long cost = waves * ((max_tiles + s - 1) / s + cost_tiles);
            if (best < 0 || cost < best) {
                best = cost;
                S = s;
            }
        }
    } else {
        S = (max_tiles + chunk_tiles - 1) / chunk_tiles;
    }
    S = std::min(std::max(S, 1l), std::min(max_tiles, 65535l));
    const long chunk = (max_tiles + S - 1) / S;
    t.chunk_tiles = (int)chunk;
    t.splits = (int)((max_tiles + chunk - 1) / chunk);
    t.ws = workspace_layout(t.splits, (size_t)B * t.q_tiles * Hkv, (size_t)total_q * Hq, D);
    return t;
}

}  // namespace pkv
