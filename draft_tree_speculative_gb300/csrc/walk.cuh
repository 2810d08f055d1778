// Greedy tree verification by one warp, shared by the walk kernel and the
// fused verify epilogue. [MI] "Walking the accepted path"; [AK] section two
// (accept_len = correct drafts + 1, the bonus is the last argmax).
//
// Each lane owns nodes `lane` and `lane + 32`. The parent and sibling rank of
// every node come from the links (or from parents), so the walk is: among the
// children of `cur` whose draft equals argmax[cur], take the lowest rank
// (first in sibling order), via one warp min-reduction per accepted level.
#pragma once

#include "common.cuh"

namespace dts {

struct WalkScratch {
  int par[kMaxNodes];
  int rank[kMaxNodes];
  int arg[kMaxNodes];
  int path[kMaxNodes];
  int nt[kMaxNodes];  // the links, staged so that following a child list reads shared memory
  int ns[kMaxNodes];
};

// Walks request b; fills ws.path[0 .. len) and ws.arg (the target argmax of
// every node) and returns len, the same in every lane. A bad link or parent
// reports and gives len = 1.
__device__ __forceinline__ int greedy_walk_warp(const int32_t *__restrict__ draft, const int32_t *__restrict__ argmax,
                                                const int32_t *__restrict__ parents,
                                                const int32_t *__restrict__ next_token,
                                                const int32_t *__restrict__ next_sibling, int b, int N,
                                                WalkScratch &ws, int lane, int32_t *err) {
  const int64_t base = static_cast<int64_t>(b) * N;
  int *par = ws.par;
  int *rank = ws.rank;
  int *arg = ws.arg;
  int *path = ws.path;
  int my_draft[2];
  for (int k = 0; k < 2; ++k) {
    const int j = lane + 32 * k;
    my_draft[k] = 0;
    if (j < N) {
      my_draft[k] = draft[base + j];
      arg[j] = argmax[base + j];
      par[j] = -2;  // "not a child of anything yet"
      rank[j] = 0;
      if (next_token != nullptr) {
        ws.nt[j] = next_token[base + j];
        ws.ns[j] = next_sibling[base + j];
      }
    }
  }
  __syncwarp();
  bool bad = false;
  if (next_token != nullptr) {
    // Each lane walks the child lists of its own nodes.
    for (int k = 0; k < 2; ++k) {
      const int p = lane + 32 * k;
      if (p >= N) continue;
      int c = ws.nt[p];
      int r = 0;
      while (c != -1) {
        if (c <= 0 || c >= N || r >= N) {  // the root is nobody's child
          bad = true;
          break;
        }
        if (atomicCAS(&par[c], -2, p) != -2) {  // a node on two lists, or a cycle
          bad = true;
          break;
        }
        rank[c] = r++;
        c = ws.ns[c];
      }
    }
  } else {
    for (int k = 0; k < 2; ++k) {
      const int j = lane + 32 * k;
      if (j >= N) continue;
      const int p = parents[base + j];
      if (j == 0 ? p != -1 : (p < 0 || p >= j)) bad = true;
      par[j] = (j == 0) ? -2 : p;
      rank[j] = j;
    }
  }
  __syncwarp();
  bad = __any_sync(0xffffffffu, bad);
  if (bad && lane == 0) report(err, next_token != nullptr ? DTS_DEV_BAD_LINK : DTS_DEV_BAD_PARENT);

  int cur = 0, len = 1;
  if (lane == 0) path[0] = 0;
  if (!bad) {
    for (int step = 1; step < N; ++step) {
      const int target = arg[cur];
      unsigned best = 0xFFFFFFFFu;
      for (int k = 0; k < 2; ++k) {
        const int j = lane + 32 * k;
        if (j < N && par[j] == cur && my_draft[k] == target)
          best = min(best, (static_cast<unsigned>(rank[j]) << 8) | static_cast<unsigned>(j));
      }
      best = __reduce_min_sync(0xffffffffu, best);
      if (best == 0xFFFFFFFFu) break;
      cur = static_cast<int>(best & 0xFFu);
      if (lane == 0) path[len] = cur;
      ++len;
    }
  }
  __syncwarp();
  return len;
}

// accept_len, the -1-padded path and the accepted tokens of request b.
__device__ __forceinline__ void write_walk_outputs(const WalkScratch &ws, int len, int b, int N, int lane,
                                                   int32_t *__restrict__ accept_len,
                                                   int32_t *__restrict__ accepted_path,
                                                   int32_t *__restrict__ accepted_tokens) {
  const int64_t base = static_cast<int64_t>(b) * N;
  for (int k = 0; k < 2; ++k) {
    const int t = lane + 32 * k;
    if (t >= N) continue;
    const int node = t < len ? ws.path[t] : -1;
    accepted_path[base + t] = node;
    accepted_tokens[base + t] = node >= 0 ? ws.arg[node] : -1;
  }
  if (lane == 0) accept_len[b] = len;
}

}  // namespace dts
