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

}  // namespace attn_sm103
