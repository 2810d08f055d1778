// Tree preparation and greedy verification.
//
// build_tree_mask: one 64-thread block per request, one thread per node.
//   [TS] "One tree attention" (64-bit ancestor mask per row), "Position follows
//   depth" (positions vc + depth), [AK] section one (a row sees itself and its
//   ancestors), [MI] "Flattening, and the two link arrays".
// verify_tree_greedy: one warp per request. [MI] "Walking the accepted path";
//   [AK] section two (accept_len = correct drafts + 1, bonus = last argmax).
#include "walk.cuh"

namespace {

using dts::kMaxNodes;

__global__ void __launch_bounds__(64) build_tree_mask_kernel(
    const int32_t *__restrict__ parents, const int32_t *__restrict__ depth,
    const int32_t *__restrict__ vc, int N, uint64_t *__restrict__ mask,
    int32_t *__restrict__ positions, int32_t *__restrict__ next_token,
    int32_t *__restrict__ next_sibling, int32_t *err) {
  __shared__ int par[kMaxNodes];
  __shared__ int dep[kMaxNodes];
  __shared__ int bad_parent, bad_depth;
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  const int64_t row = static_cast<int64_t>(b) * N + i;
  if (i == 0) {
    bad_parent = 0;
    bad_depth = 0;
  }
  if (i < N) {
    par[i] = parents[row];
    dep[i] = depth[row];
  }
  __syncthreads();
  if (i < N) {
    const int p = par[i];
    if (i == 0) {
      if (p != -1) bad_parent = 1;
      else if (dep[0] != 0) bad_depth = 1;
    } else if (p < 0 || p >= i) {
      bad_parent = 1;
    } else if (dep[i] != dep[p] + 1) {
      bad_depth = 1;
    }
  }
  __syncthreads();
  if (i >= N) return;
  const int v = vc[b];
  if (bad_parent | bad_depth) {
    if (i == 0) dts::report(err, bad_parent ? DTS_DEV_BAD_PARENT : DTS_DEV_BAD_DEPTH);
    mask[row] = 0;
    positions[row] = v;
    next_token[row] = -1;
    next_sibling[row] = -1;
    return;
  }
  // Ancestor walk: parents[j] < j, so this ends within i + 1 steps.
  uint64_t m = 0;
  for (int j = i; j >= 0; j = par[j]) m |= 1ull << j;
  int first_child = -1, sibling = -1;
  for (int j = N - 1; j > i; --j) {       // lowest index wins: scan downwards
    if (par[j] == i) first_child = j;
    if (i > 0 && par[j] == par[i]) sibling = j;
  }
  mask[row] = m;
  positions[row] = v + dep[i];
  next_token[row] = first_child;
  next_sibling[row] = sibling;
}

// One warp per request (the walk itself in walk.cuh).
__global__ void __launch_bounds__(128) verify_tree_greedy_kernel(
    const int32_t *__restrict__ draft, const int32_t *__restrict__ argmax,
    const int32_t *__restrict__ parents, const int32_t *__restrict__ next_token,
    const int32_t *__restrict__ next_sibling, int B, int N, int32_t *__restrict__ accept_len,
    int32_t *__restrict__ accepted_path, int32_t *__restrict__ accepted_tokens, int32_t *err) {
  constexpr int kWarps = 4;
  __shared__ dts::WalkScratch s_walk[kWarps];
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarps + w;
  if (b >= B) return;
  const int len = dts::greedy_walk_warp(draft, argmax, parents, next_token, next_sibling, b, N, s_walk[w], lane, err);
  dts::write_walk_outputs(s_walk[w], len, b, N, lane, accept_len, accepted_path, accepted_tokens);
}

}  // namespace

extern "C" int dts_build_tree_mask(const int32_t *parents, const int32_t *depth, const int32_t *vc,
                                   int B, int N, uint64_t *mask, int32_t *positions,
                                   int32_t *next_token, int32_t *next_sibling, int32_t *err_dev,
                                   dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0) return DTS_OK;
  if (!parents || !depth || !vc || !mask || !positions || !next_token || !next_sibling)
    return DTS_ERR_INVALID;
  build_tree_mask_kernel<<<B, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      parents, depth, vc, N, mask, positions, next_token, next_sibling, err_dev);
  return dts_host::launch_status();
}

extern "C" int dts_verify_tree_greedy(const int32_t *draft_tokens, const int32_t *target_argmax,
                                      const int32_t *parents, const int32_t *next_token,
                                      const int32_t *next_sibling, int B, int N,
                                      int32_t *accept_len, int32_t *accepted_path,
                                      int32_t *accepted_tokens, int32_t *err_dev,
                                      dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0) return DTS_OK;
  if (!draft_tokens || !target_argmax || !accept_len || !accepted_path || !accepted_tokens)
    return DTS_ERR_INVALID;
  if ((next_token == nullptr) != (next_sibling == nullptr)) return DTS_ERR_INVALID;
  if (next_token == nullptr && parents == nullptr) return DTS_ERR_INVALID;
  const int blocks = (B + 3) / 4;
  verify_tree_greedy_kernel<<<blocks, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      draft_tokens, target_argmax, parents, next_token, next_sibling, B, N, accept_len,
      accepted_path, accepted_tokens, err_dev);
  return dts_host::launch_status();
}
