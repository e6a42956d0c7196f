// sv_treemask.cuh -- the tree-attention mask and depth position ids of a
// depth-first linearised token tree.
//
// Tree attention (CMU 15-779 Lecture 17 notes, "Speculative Decoding",
// sec. 4.3): the tree is laid out depth first, ancestors before their
// descendants; a node attends to the verified prefix, to its own ancestors
// and to itself, and takes its position from its depth, so nodes at one
// depth share a position (sec. 10 exercise 5 works one tree through).
//
// One warp per request.  The parents (at most 64 nodes) go to shared
// memory; lane l owns nodes l and l + 32 and climbs from each to the root,
// setting one mask bit per node passed.  Each climb is at most 63 steps and
// reads only shared memory; the whole tree is validated first (parent[0]
// == -1, 0 <= parent[i] < i), so every climb ends.
#pragma once

#include "sv_rowpass.cuh"

namespace sv {

constexpr int kMaskWarps = 8;  // requests per CTA

struct MaskProblem {
  int B, N, words;
  const int* parent;
  const int* num_nodes;
  unsigned* mask;
  int* depth;
  WsHeader* hdr;
};

__global__ void __launch_bounds__(kMaskWarps * 32) tree_mask_kernel(const MaskProblem a) {
  __shared__ int par_s[kMaskWarps][SV_MAX_TREE_NODES];
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int b = static_cast<int>(blockIdx.x) * kMaskWarps + warp;
  if (b >= a.B) return;
  const int N = a.N;
  const int n = a.num_nodes ? a.num_nodes[b] : N;
  int* par = par_s[warp];
  const bool n_ok = n >= 1 && n <= N;
  bool bad = false;
  for (int i = lane; i < N; i += 32) {
    const int p = a.parent[static_cast<size_t>(b) * N + i];
    par[i] = p;
    if (n_ok && i < n) bad |= i == 0 ? p != -1 : (p < 0 || p >= i);
  }
  const bool tree_bad = __any_sync(0xffffffffu, bad);
  __syncwarp();
  const bool ok = n_ok && !tree_bad;
  if (lane == 0 && !ok) record_error(&a.hdr->error, n_ok ? SV_DERR_TREE : SV_DERR_ARG);
  for (int i = lane; i < N; i += 32) {
    unsigned long long bits = 0ull;
    int d = -1;
    if (ok && i < n) {
      for (int j = i; j >= 0; j = j == 0 ? -1 : par[j]) {
        bits |= 1ull << j;
        ++d;
      }
    }
    unsigned* row = a.mask + (static_cast<size_t>(b) * N + i) * a.words;
    for (int w = 0; w < a.words; ++w)
      row[w] = w < 2 ? static_cast<unsigned>(bits >> (32 * w)) : 0u;
    a.depth[static_cast<size_t>(b) * N + i] = d;
  }
}

}  // namespace sv
