// CTA order of the causal grids, per kernel and kernel width: the longest-first
// (tile-major) order is used when the bytes that the blocks of one head share, summed
// over all heads, are at most max_tile_major_bytes; otherwise each head's blocks run
// together. Written by tune_grid_order.py from a timing sweep of both orders on causal
// dense inputs on a GB300 (NVIDIA GB300); regenerate, do not edit.
#pragma once

namespace attn_sm103 {

struct GridOrderRule {
  const char* kernel;
  int width;
  double max_tile_major_bytes;
};

static const GridOrderRule kGridOrderRules[] = {
    {"fwd", 64, 134217728.0},  // mean slowdown 1.0006 over 10 points
    {"fwd", 128, 134217728.0},  // mean slowdown 1.0003 over 10 points
    {"bwd_main", 64, 67108864.0},  // mean slowdown 1.0000 over 10 points
    {"bwd_main", 128, 134217728.0},  // mean slowdown 1.0000 over 10 points
    {"bwd_main_nodq", 64, 33554432.0},  // mean slowdown 1.0007 over 10 points
    {"bwd_main_nodq", 128, 67108864.0},  // mean slowdown 1.0000 over 10 points
    {"bwd_dq", 64, 134217728.0},  // mean slowdown 1.0002 over 10 points
    {"bwd_dq", 128, 67108864.0},  // mean slowdown 1.0006 over 10 points
};

// Split key ranges of a non-causal dense forward, per kernel width: used when the
// query blocks are at most max_blocks_per_sm x the SM count (and at most half of
// it, so that every block has the same number of parts) and each block has at
// least min_key_tiles key tiles. Written by tune_grid_order.py --split from a
// timing sweep of the forward with and without the split on a GB300 (NVIDIA GB300).
struct FwdSplitRule {
  int width;
  double max_blocks_per_sm;
  int min_key_tiles;
};

static const FwdSplitRule kFwdSplitRules[] = {
    {64, 0.500000, 16},  // mean slowdown 1.0022 over 30 points
    {128, 0.500000, 16},  // mean slowdown 1.0054 over 30 points
    {256, 0.473684, 32},  // mean slowdown 1.0071 over 30 points
};

}  // namespace attn_sm103
