// Compaction entry points: the path's KV rows in every buffer of a cache
// group's address table, and the hidden rows plus positions (the work itself
// in compact.cuh).
#include "compact.cuh"

namespace {

using dts::kBufPerBlock;
using dts::kThreads;

// grid (ceil(n_buffers / kBufPerBlock), B)
__global__ void __launch_bounds__(kThreads) compact_window_rows_kernel(
    const dts_kv_buffer *__restrict__ table, int n_buffers, const int64_t *__restrict__ wl,
    const int32_t *__restrict__ accepted_path, const int32_t *__restrict__ accept_len, int N, int32_t *err) {
  __shared__ dts::KvCompactSmem kv;
  const int b = blockIdx.y;
  dts::kv_prepare(table, n_buffers, blockIdx.x, wl, b, N, kv, threadIdx.x, kThreads);
  __syncthreads();
  dts::kv_move(n_buffers, blockIdx.x, accepted_path + static_cast<int64_t>(b) * N, accept_len[b], b, N, kv, err);
}

// grid (B)
__global__ void __launch_bounds__(kThreads) compact_rows_kernel(
    char *__restrict__ hidden, int64_t row_bytes, int32_t *__restrict__ positions, const int32_t *__restrict__ vc,
    const int32_t *__restrict__ accepted_path, const int32_t *__restrict__ accept_len, int N, int32_t *err) {
  const int b = blockIdx.x;
  dts::write_positions(positions, vc, b, N, threadIdx.x, kThreads);
  dts::move_hidden_block(hidden, row_bytes, accepted_path + static_cast<int64_t>(b) * N,
                         hidden != nullptr ? accept_len[b] : 0, b, N, err);
}

}  // namespace

extern "C" int dts_compact_window_rows(const dts_kv_buffer *table, int n_buffers,
                                       const int64_t *write_locations, const int32_t *accepted_path,
                                       const int32_t *accept_len, int B, int N, int32_t *err_dev,
                                       dts_stream_t stream) {
  if (B < 0 || N < 1 || n_buffers < 0) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0 || n_buffers == 0) return DTS_OK;
  if (n_buffers > 65535 || B > 65535) return DTS_ERR_UNSUPPORTED;
  if (!table || !write_locations || !accepted_path || !accept_len) return DTS_ERR_INVALID;
  const int groups = (n_buffers + kBufPerBlock - 1) / kBufPerBlock;
  compact_window_rows_kernel<<<dim3(groups, B), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      table, n_buffers, write_locations, accepted_path, accept_len, N, err_dev);
  return dts_host::launch_status();
}

extern "C" int dts_compact_rows(void *hidden, int64_t row_bytes, int32_t *positions, const int32_t *vc,
                                const int32_t *accepted_path, const int32_t *accept_len, int B, int N,
                                int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0 || (hidden == nullptr && positions == nullptr)) return DTS_OK;
  if (hidden != nullptr && (row_bytes <= 0 || (row_bytes & 3) != 0 || row_bytes > (1ll << 30) ||
                            (reinterpret_cast<uintptr_t>(hidden) & 3) != 0))
    return DTS_ERR_INVALID;
  if (hidden != nullptr && (!accepted_path || !accept_len)) return DTS_ERR_INVALID;
  if (positions != nullptr && vc == nullptr) return DTS_ERR_INVALID;
  compact_rows_kernel<<<B, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<char *>(hidden), row_bytes, positions, vc, accepted_path, accept_len, N, err_dev);
  return dts_host::launch_status();
}
