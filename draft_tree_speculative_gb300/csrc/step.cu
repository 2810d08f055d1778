// The verify step's small stages fused into two launches around the
// attention:
//
//   prologue: build_tree_mask and write_window_kv, one warp per node. The
//             warp reads its request's tree (lane l holds nodes l and l + 32),
//             validates it, forms its node's ancestor mask by walking the
//             parents with shuffles, its first child and next sibling by
//             ballots, its position vc + depth, and then writes the node's
//             rotated K and its V (window_kv.cuh).
//   epilogue: verify_tree_greedy, compact_window_rows and compact_rows, one
//             block per (request, group of KV buffers). Warp 0 walks the tree
//             (walk.cuh) into shared memory, and the block compacts that
//             request's rows along the path (compact.cuh).
//
// Each produces exactly what the separate calls produce (the same device code
// does the work); only the launches and the round trips through global
// memory between them go. Sources as for the separate calls: [TS] "One tree
// attention", "Position follows depth, slot follows node index", "The tree is
// a parameter of the chain path"; [AK] sections one and two; [MI] "Building
// the mask, for real", "Flattening, and the two link arrays", "Walking the
// accepted path", "Discarding the rejected branches' KV".
#include "compact.cuh"
#include "walk.cuh"
#include "window_kv.cuh"

namespace {

struct PrologueArgs {
  dts::WindowKvArgs kv;  // (kv.positions is not read: the position comes from the tree)
  const int32_t *parents, *depth, *vc;
  uint64_t *mask;
  int32_t *positions, *next_token, *next_sibling;
};

// Node j's value of a per-node pair held as (lane j, lane j - 32): v0 in lane
// j for j < 32, v1 in lane j - 32 otherwise. `j` may differ between lanes.
__device__ __forceinline__ int node_value(int v0, int v1, int j) {
  const int x0 = __shfl_sync(0xffffffffu, v0, j & 31);
  const int x1 = __shfl_sync(0xffffffffu, v1, j & 31);
  return j < 32 ? x0 : x1;
}

template <int D>
__global__ void __launch_bounds__(256) verify_prologue_kernel(const __grid_constant__ PrologueArgs a) {
  dts::grid_dep_wait();
  dts::grid_dep_launch_next();
  const int node = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // b * N + i
  const int lane = threadIdx.x & 31;
  const int B = a.kv.B, N = a.kv.N;
  if (node >= B * N) return;
  const int b = node / N;
  const int i = node - b * N;
  const int64_t base = static_cast<int64_t>(b) * N;
  const int j0 = lane, j1 = lane + 32;
  const int p0 = j0 < N ? a.parents[base + j0] : 0, d0 = j0 < N ? a.depth[base + j0] : 0;
  const int p1 = j1 < N ? a.parents[base + j1] : 0, d1 = j1 < N ? a.depth[base + j1] : 0;
  // the checks of build_tree_mask: a bad parent anywhere wins over a bad depth
  bool bad_par = false, bad_dep = false;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int j = k == 0 ? j0 : j1;
    const int p = k == 0 ? p0 : p1;
    const int dj = k == 0 ? d0 : d1;
    const bool pok = j == 0 ? p == -1 : (p >= 0 && p < j);
    const int dp = node_value(d0, d1, pok && j > 0 ? p : 0);  // (every lane takes part in the shuffle)
    if (j < N) {
      if (!pok) bad_par = true;
      else if (j == 0 ? dj != 0 : dj != dp + 1) bad_dep = true;
    }
  }
  bad_par = __any_sync(0xffffffffu, bad_par);
  bad_dep = __any_sync(0xffffffffu, bad_dep);
  const int v = a.vc[b];
  int pos = v;
  if (bad_par || bad_dep) {
    if (lane == 0) {
      if (i == 0) dts::report(a.kv.err, bad_par ? DTS_DEV_BAD_PARENT : DTS_DEV_BAD_DEPTH);
      a.mask[node] = 0;
      a.positions[node] = v;
      a.next_token[node] = -1;
      a.next_sibling[node] = -1;
    }
  } else {
    // ancestor walk: parents[j] < j, so it ends within i + 1 steps
    uint64_t m = 0;
    for (int j = i; j >= 0; j = node_value(p0, p1, j)) m |= 1ull << j;
    const int pi = node_value(p0, p1, i);
    // the lowest-index child and the next higher-index sibling
    const uint32_t c0 = __ballot_sync(0xffffffffu, j0 < N && j0 > i && p0 == i);
    const uint32_t c1 = __ballot_sync(0xffffffffu, j1 < N && j1 > i && p1 == i);
    const uint32_t s0 = __ballot_sync(0xffffffffu, i > 0 && j0 < N && j0 > i && p0 == pi);
    const uint32_t s1 = __ballot_sync(0xffffffffu, i > 0 && j1 < N && j1 > i && p1 == pi);
    const int first_child = c0 ? __ffs(c0) - 1 : (c1 ? 31 + __ffs(c1) : -1);
    const int sibling = s0 ? __ffs(s0) - 1 : (s1 ? 31 + __ffs(s1) : -1);
    pos = v + node_value(d0, d1, i);
    if (lane == 0) {
      a.mask[node] = m;
      a.positions[node] = pos;
      a.next_token[node] = first_child;
      a.next_sibling[node] = sibling;
    }
  }
  dts::write_node_kv<D, false>(a.kv, node, pos, lane);
}

struct EpilogueArgs {
  const int32_t *draft, *argmax, *parents, *next_token, *next_sibling;
  int32_t *accept_len, *accepted_path, *accepted_tokens;
  const dts_kv_buffer *table;
  int n_buffers;
  const int64_t *write_locations;
  char *hidden;
  int64_t row_bytes;
  int32_t *positions;
  const int32_t *vc;
  int32_t *err;
  int N;
  int kv_groups;  // blocks per request that move KV rows
};

// grid (kv_groups + 1, B). Every block walks request b with warp 0 (the path
// lands in shared memory). Meanwhile the other warps of block gx < kv_groups
// stage what the KV move of buffer group gx needs short of the path (the
// entries, their checks, the window slots), and those of the last block write
// the positions; then block gx moves its KV rows, and the last block writes the
// walk's outputs and moves the hidden rows.
__global__ void __launch_bounds__(dts::kThreads) verify_epilogue_kernel(const __grid_constant__ EpilogueArgs a) {
  dts::grid_dep_wait();
  dts::grid_dep_launch_next();
  __shared__ dts::WalkScratch ws;
  __shared__ dts::KvCompactSmem kv;
  __shared__ int s_len;
  const int b = blockIdx.y, gx = blockIdx.x;
  const bool rows_block = gx == a.kv_groups;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int len =
        dts::greedy_walk_warp(a.draft, a.argmax, a.parents, a.next_token, a.next_sibling, b, a.N, ws, lane, a.err);
    if (rows_block)
      dts::write_walk_outputs(ws, len, b, a.N, lane, a.accept_len, a.accepted_path, a.accepted_tokens);
    if (lane == 0) s_len = len;
  } else if (!rows_block) {
    dts::kv_prepare(a.table, a.n_buffers, gx, a.write_locations, b, a.N, kv, threadIdx.x - 32, dts::kThreads - 32);
  } else {
    dts::write_positions(a.positions, a.vc, b, a.N, threadIdx.x - 32, dts::kThreads - 32);
  }
  __syncthreads();
  const int alen = s_len;
  if (!rows_block) dts::kv_move(a.n_buffers, gx, ws.path, alen, b, a.N, kv, a.err);
  else dts::move_hidden_block(a.hidden, a.row_bytes, ws.path, alen, b, a.N, a.err);
}

}  // namespace

extern "C" int dts_verify_prologue(const int32_t *parents, const int32_t *depth, const int32_t *vc,
                                   const uint16_t *k_new, const uint16_t *v_new, const int32_t *page_table,
                                   int max_pages, int page_size, const int32_t *prefix_len, int B, int N, int Hkv,
                                   int d, int64_t num_slots, float rope_theta, uint64_t *mask, int32_t *positions,
                                   int32_t *next_token, int32_t *next_sibling, uint16_t *k_cache, uint16_t *v_cache,
                                   int64_t *write_locations, int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1 || Hkv < 1 || max_pages < 1 || num_slots < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes || (d != 64 && d != 128)) return DTS_ERR_UNSUPPORTED;
  if (page_size < 8 || page_size > 4096 || (page_size & (page_size - 1)) != 0) return DTS_ERR_UNSUPPORTED;
  if (!(rope_theta > 0.f)) return DTS_ERR_INVALID;
  if (B == 0) return DTS_OK;
  if (!parents || !depth || !vc || !k_new || !v_new || !page_table || !prefix_len || !mask || !positions ||
      !next_token || !next_sibling || !k_cache || !v_cache)
    return DTS_ERR_INVALID;
  const uintptr_t al = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
  if (al & 7) return DTS_ERR_INVALID;
  PrologueArgs a;
  a.kv.k_new = k_new;
  a.kv.v_new = v_new;
  a.kv.positions = nullptr;
  a.kv.page_table = page_table;
  a.kv.prefix_len = prefix_len;
  a.kv.k_cache = k_cache;
  a.kv.v_cache = v_cache;
  a.kv.write_locations = write_locations;
  a.kv.err = err_dev;
  a.kv.num_slots = num_slots;
  a.kv.max_pages = max_pages;
  a.kv.page_shift = __builtin_ctz(static_cast<unsigned>(page_size));
  a.kv.B = B;
  a.kv.N = N;
  a.kv.Hkv = Hkv;
  dts_host::make_rope_freqs(rope_theta, d, &a.kv.freqs);
  a.parents = parents;
  a.depth = depth;
  a.vc = vc;
  a.mask = mask;
  a.positions = positions;
  a.next_token = next_token;
  a.next_sibling = next_sibling;
  const int64_t warps = static_cast<int64_t>(B) * N;
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d == 128) dts_host::launch_chained(verify_prologue_kernel<128>, dim3(blocks), dim3(256), 0, s, a);
  else dts_host::launch_chained(verify_prologue_kernel<64>, dim3(blocks), dim3(256), 0, s, a);
  return dts_host::launch_status();
}

extern "C" int dts_verify_epilogue(const int32_t *draft_tokens, const int32_t *target_argmax,
                                   const int32_t *parents, const int32_t *next_token, const int32_t *next_sibling,
                                   int B, int N, int32_t *accept_len, int32_t *accepted_path,
                                   int32_t *accepted_tokens, const dts_kv_buffer *table, int n_buffers,
                                   const int64_t *write_locations, void *hidden, int64_t row_bytes,
                                   int32_t *positions, const int32_t *vc, int32_t *err_dev, dts_stream_t stream) {
  // the checks of dts_verify_tree_greedy, dts_compact_window_rows and dts_compact_rows
  if (B < 0 || N < 1 || n_buffers < 0) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0) return DTS_OK;
  if (n_buffers > 65535 || B > 65535) return DTS_ERR_UNSUPPORTED;
  if (!draft_tokens || !target_argmax || !accept_len || !accepted_path || !accepted_tokens) return DTS_ERR_INVALID;
  if ((next_token == nullptr) != (next_sibling == nullptr)) return DTS_ERR_INVALID;
  if (next_token == nullptr && parents == nullptr) return DTS_ERR_INVALID;
  if (n_buffers > 0 && (!table || !write_locations)) return DTS_ERR_INVALID;
  if (hidden != nullptr && (row_bytes <= 0 || (row_bytes & 3) != 0 || row_bytes > (1ll << 30) ||
                            (reinterpret_cast<uintptr_t>(hidden) & 3) != 0))
    return DTS_ERR_INVALID;
  if (positions != nullptr && vc == nullptr) return DTS_ERR_INVALID;
  EpilogueArgs a;
  a.draft = draft_tokens;
  a.argmax = target_argmax;
  a.parents = parents;
  a.next_token = next_token;
  a.next_sibling = next_sibling;
  a.accept_len = accept_len;
  a.accepted_path = accepted_path;
  a.accepted_tokens = accepted_tokens;
  a.table = table;
  a.n_buffers = n_buffers;
  a.write_locations = write_locations;
  a.hidden = static_cast<char *>(hidden);
  a.row_bytes = row_bytes;
  a.positions = positions;
  a.vc = vc;
  a.err = err_dev;
  a.N = N;
  a.kv_groups = (n_buffers + dts::kBufPerBlock - 1) / dts::kBufPerBlock;
  dts_host::launch_chained(verify_epilogue_kernel, dim3(a.kv_groups + 1, B), dim3(dts::kThreads), 0,
                           reinterpret_cast<cudaStream_t>(stream), a);
  return dts_host::launch_status();
}
