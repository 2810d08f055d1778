// The target's argmax at every verify row, and the greedy walk fed by it.
//
// [MI] "Walking the accepted path": target_predict is the target's argmax at
// each node's position, computed for all nodes by the one verify forward; the
// walk compares the draft tokens against it. [MI], the worked (5, 4, 8)
// iteration, step 5: the argmax over all rows is taken, then the tree walked.
//
// The logits [rows][vocab] fp32 are read once, so the pass is bound by HBM.
// Two kernels:
//
// 1. argmax_chunk_kernel: one block per (row, chunk of 16384 logits). Every
//    thread issues all of its loads first (16 float4 per thread, consecutive
//    threads on consecutive 16-byte words), then keeps the best (value, index)
//    of its elements; the block's best goes to the workspace as one packed
//    64-bit word.
// 2. argmax_reduce_kernel: one thread per row takes the largest of the row's
//    chunk words and writes the int32 index.
//
// Order: a float maps to a 32-bit key that orders like the value (sign-magnitude
// folded to unsigned), with every NaN mapped above +inf and -0 mapped onto +0;
// the packed word is (key << 32) | ~index, so the largest word holds the
// largest value and, among equal values, the lowest index. These are NumPy's
// argmax rules: ties to the lowest index, the first NaN wins, -0 == +0.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 16;                     // float4 loads per thread
constexpr int kChunk = kThreads * kVec * 4;  // logits per block

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;  // NaN: above every number
  if (b == 0x80000000u) b = 0u;                              // -0 equals +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint64_t packed(float x, uint32_t index) {
  return (static_cast<uint64_t>(order_key(x)) << 32) | static_cast<uint32_t>(~index);
}

// The block's best packed word over elements [lo, hi) of a row (0 if empty:
// below every packed word, whose key is at least that of -inf).
__device__ __forceinline__ uint64_t block_max(uint64_t b) {
  __shared__ uint64_t part[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t x = __shfl_xor_sync(0xffffffffu, b, o);
    b = x > b ? x : b;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) part[warp] = b;
  __syncthreads();
  if (warp == 0) {
    b = lane < kThreads / 32 ? part[lane] : 0ull;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      const uint64_t x = __shfl_xor_sync(0xffffffffu, b, o);
      b = x > b ? x : b;
    }
  }
  return b;
}

// A thread's running best over elements it visits in increasing index order:
// a later element replaces it only if strictly larger, or a NaN over a
// number, so among equal values (and among NaNs) the first stays. -0 and +0
// compare equal as floats.
struct Best {
  float v = -INFINITY;
  int i = -1;  // -1: no element seen yet
  __device__ __forceinline__ void see(float x, int idx) {
    const bool take = x > v || (x != x && v == v) || i < 0;
    v = take ? x : v;
    i = take ? idx : i;
  }
  __device__ __forceinline__ uint64_t word() const { return i < 0 ? 0ull : packed(v, static_cast<uint32_t>(i)); }
};

// kVec4: the row starts on a 16-byte boundary (logits aligned, row stride a
// multiple of 4), so whole float4 words inside the row are read as such.
template <bool kVec4>
__global__ void __launch_bounds__(kThreads) argmax_chunk_kernel(const float *logits, int64_t row_stride, int vocab,
                                                                int chunks, uint64_t *best) {
  const int64_t blk = blockIdx.x;
  const int64_t row = blk / chunks;
  const int c = static_cast<int>(blk - row * chunks);
  const float *src = logits + row * row_stride;
  const int lo = c * kChunk;
  const int hi = min(vocab, lo + kChunk);
  const int tid = static_cast<int>(threadIdx.x);
  Best bt;
  if (kVec4 && hi - lo == kChunk) {
    // a whole chunk: every load issued first, no bounds to test
    float4 v[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) v[k] = __ldcs(reinterpret_cast<const float4 *>(src + lo) + k * kThreads + tid);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int e = lo + (k * kThreads + tid) * 4;
      bt.see(v[k].x, e);
      bt.see(v[k].y, e + 1);
      bt.see(v[k].z, e + 2);
      bt.see(v[k].w, e + 3);
    }
  } else if (kVec4) {
    // the row's last chunk: whole float4 words, then the ragged end
    for (int e = lo + tid * 4; e < hi; e += kThreads * 4) {
      if (e + 4 <= hi) {
        const float4 x = __ldcs(reinterpret_cast<const float4 *>(src + e));
        bt.see(x.x, e);
        bt.see(x.y, e + 1);
        bt.see(x.z, e + 2);
        bt.see(x.w, e + 3);
      } else {
        for (int q = e; q < hi; ++q) bt.see(src[q], q);
      }
    }
  } else {
    for (int e = lo + tid; e < hi; e += kThreads) bt.see(src[e], e);
  }
  const uint64_t b = block_max(bt.word());
  if (threadIdx.x == 0) best[blk] = b;
}

__global__ void __launch_bounds__(256) argmax_reduce_kernel(const uint64_t *best, int64_t rows, int chunks,
                                                            int32_t *argmax) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= rows) return;
  uint64_t b = 0ull;
  for (int c = 0; c < chunks; ++c) {
    const uint64_t x = best[row * chunks + c];
    b = x > b ? x : b;
  }
  argmax[row] = static_cast<int32_t>(~static_cast<uint32_t>(b));
}

int chunks_of(int vocab) { return (vocab + kChunk - 1) / kChunk; }

}  // namespace

extern "C" size_t dts_target_argmax_workspace(int64_t rows, int vocab) {
  if (rows < 0 || vocab < 1) return 0;
  return static_cast<size_t>(rows) * chunks_of(vocab) * sizeof(uint64_t);
}

extern "C" int dts_target_argmax(const float *logits, int64_t rows, int vocab, int64_t row_stride, int32_t *argmax,
                                 void *workspace, size_t ws_bytes, dts_stream_t stream) {
  if (rows < 0 || vocab < 1 || row_stride < vocab) return DTS_ERR_INVALID;
  if (rows == 0) return DTS_OK;
  if (!logits || !argmax || (reinterpret_cast<uintptr_t>(logits) & 3)) return DTS_ERR_INVALID;
  const int chunks = chunks_of(vocab);
  if (rows * chunks >= (1ll << 31)) return DTS_ERR_UNSUPPORTED;
  if (workspace == nullptr || ws_bytes < dts_target_argmax_workspace(rows, vocab)) return DTS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 7) return DTS_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint64_t *best = static_cast<uint64_t *>(workspace);
  const unsigned blocks = static_cast<unsigned>(rows * chunks);
  const bool vec4 = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && (row_stride & 3) == 0;
  if (vec4) argmax_chunk_kernel<true><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best);
  else argmax_chunk_kernel<false><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best);
  if (dts_host::launch_status() != DTS_OK) return DTS_ERR_CUDA;
  argmax_reduce_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(best, rows, chunks, argmax);
  return dts_host::launch_status();
}

extern "C" int dts_verify_tree_greedy_logits(const int32_t *draft_tokens, const float *logits, int vocab,
                                             int64_t row_stride, const int32_t *parents, const int32_t *next_token,
                                             const int32_t *next_sibling, int B, int N, int32_t *target_argmax,
                                             int32_t *accept_len, int32_t *accepted_path, int32_t *accepted_tokens,
                                             void *workspace, size_t ws_bytes, int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0) return DTS_OK;
  if (!draft_tokens || !target_argmax || !accept_len || !accepted_path || !accepted_tokens) return DTS_ERR_INVALID;
  if ((next_token == nullptr) != (next_sibling == nullptr)) return DTS_ERR_INVALID;
  if (next_token == nullptr && parents == nullptr) return DTS_ERR_INVALID;
  const int st = dts_target_argmax(logits, static_cast<int64_t>(B) * N, vocab, row_stride, target_argmax, workspace,
                                   ws_bytes, stream);
  if (st != DTS_OK) return st;
  return dts_verify_tree_greedy(draft_tokens, target_argmax, parents, next_token, next_sibling, B, N, accept_len,
                                accepted_path, accepted_tokens, err_dev, stream);
}
