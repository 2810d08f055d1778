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

// Sampled draws ([TS] "Sampled verify keys noise by position"): the same pass
// with each logit x of row (b, i) replaced by x * (1/T_b) + G(seed_b, pos, v),
// pos = vc_b + depth[b][i] + 1, G Gumbel noise; the row's argmax is its draw.
// The noise and its float32 arithmetic are fixed exactly (one IEEE rounding
// per operation, no fused multiply-add) so that the draw is reproducible:
//   words: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
//          as easy as 1, 2, 3", SC 2011), key (seed low, seed high), counter
//          (v / 4, pos, 0, 0), word v % 4 for vocabulary entry v;
//   u = (2 (word >> 9) + 1) 2^-24, exact, in (0, 1);
//   G = -ln(-ln u), ln as log_f32 below.
// T_b <= 0 or not finite: no noise (the plain argmax).

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

struct Words {
  uint32_t w[4];
};

// Philox4x32-10: ten rounds of two 32x32->64 multiplies; the key is bumped by
// the Weyl constants before every round but the first.
__device__ __forceinline__ Words philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return Words{{c0, c1, c2, c3}};
}

// ln x for positive normal x: x = m 2^e with m in [1, 2), halved (e + 1) above
// sqrt 2; s = (m - 1)/(m + 1); ln m = 2 atanh s = 2 s (1 + t/3 + t^2/5 + t^3/7
// + t^4/9), t = s^2, |s| <= 0.1716 (the dropped terms are below 4e-10
// relative); ln x = e ln 2 + ln m. Coefficients are the float32 roundings of
// 1/3, 1/5, 1/7, 1/9, ln 2 and sqrt 2; every operation is rounded once.
__device__ __forceinline__ float log_f32(float x) {
  const float kLn2 = 0x1.62e430p-1f, kSqrt2 = 0x1.6a09e6p+0f;
  const float kC3 = 0x1.555556p-2f, kC5 = 0x1.99999ap-3f, kC7 = 0x1.24924ap-3f, kC9 = 0x1.c71c72p-4f;
  const uint32_t b = __float_as_uint(x);
  int e = static_cast<int>((b >> 23) & 0xFFu) - 127;
  float m = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
  if (m > kSqrt2) {
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float t = __fmul_rn(s, s);
  float p = __fmul_rn(t, kC9);
  p = __fmul_rn(__fadd_rn(p, kC7), t);
  p = __fmul_rn(__fadd_rn(p, kC5), t);
  p = __fmul_rn(__fadd_rn(p, kC3), t);
  p = __fadd_rn(p, 1.0f);
  return __fadd_rn(__fmul_rn(static_cast<float>(e), kLn2), __fmul_rn(__fadd_rn(s, s), p));
}

__device__ __forceinline__ float gumbel(uint32_t word) {
  const float u = __fmul_rn(static_cast<float>((word >> 9) * 2u + 1u), 0x1p-24f);
  return -log_f32(-log_f32(u));
}

// Per-row sampling parameters (all device arrays): row r = b*N + i.
struct Sampler {
  const int32_t *vc;       // [B]
  const int32_t *depth;    // [B][N]
  const float *temperature;  // [B]
  const uint64_t *seed;    // [B]
  int N;
};

struct RowNoise {
  bool on;
  float inv_t;
  uint32_t pos, k0, k1;
  __device__ __forceinline__ float score(float x, const Words &w, int q) const {
    return __fadd_rn(__fmul_rn(x, inv_t), gumbel(w.w[q]));
  }
  __device__ __forceinline__ Words words(int v4) const { return philox4x32_10(static_cast<uint32_t>(v4), pos, 0u, 0u, k0, k1); }
};

__device__ __forceinline__ RowNoise row_noise(const Sampler &sp, int64_t row) {
  RowNoise rn;
  const int64_t b = row / sp.N;
  const float t = sp.temperature[b];
  rn.on = t > 0.f && t <= 3.402823466e38f;  // finite and positive
  rn.inv_t = rn.on ? __fdiv_rn(1.0f, t) : 1.0f;
  rn.pos = static_cast<uint32_t>(sp.vc[b] + sp.depth[row] + 1);
  const uint64_t seed = sp.seed[b];
  rn.k0 = static_cast<uint32_t>(seed);
  rn.k1 = static_cast<uint32_t>(seed >> 32);
  return rn;
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
template <bool kVec4, bool kSample>
__global__ void __launch_bounds__(kThreads, kSample ? 6 : 1) argmax_chunk_kernel(const float *logits, int64_t row_stride, int vocab,
                                                                int chunks, uint64_t *best, Sampler sp) {
  const int64_t blk = blockIdx.x;
  const int64_t row = blk / chunks;
  const int c = static_cast<int>(blk - row * chunks);
  const float *src = logits + row * row_stride;
  const int lo = c * kChunk;
  const int hi = min(vocab, lo + kChunk);
  const int tid = static_cast<int>(threadIdx.x);
  Best bt;
  RowNoise rn;
  if (kSample) rn = row_noise(sp, row);
  // the element's score: the logit, or its sampled score
  auto see4 = [&](const float4 &x, int e) {
    if (kSample && rn.on) {
      const Words w = rn.words(e >> 2);
      bt.see(rn.score(x.x, w, 0), e);
      bt.see(rn.score(x.y, w, 1), e + 1);
      bt.see(rn.score(x.z, w, 2), e + 2);
      bt.see(rn.score(x.w, w, 3), e + 3);
    } else {
      bt.see(x.x, e);
      bt.see(x.y, e + 1);
      bt.see(x.z, e + 2);
      bt.see(x.w, e + 3);
    }
  };
  auto see1 = [&](float x, int e) {
    if (kSample && rn.on) bt.see(rn.score(x, rn.words(e >> 2), e & 3), e);
    else bt.see(x, e);
  };
  if (kVec4 && hi - lo == kChunk) {
    // a whole chunk, no bounds to test. The plain argmax is bound by HBM: every
    // load is issued first. The sampled scores are bound by arithmetic: four
    // loads at a time keep the registers (and so the warps per SM) for it.
    constexpr int kDepth = kSample ? 4 : kVec;
#pragma unroll
    for (int k0 = 0; k0 < kVec; k0 += kDepth) {
      float4 v[kDepth];
#pragma unroll
      for (int k = 0; k < kDepth; ++k)
        v[k] = __ldcs(reinterpret_cast<const float4 *>(src + lo) + (k0 + k) * kThreads + tid);
#pragma unroll
      for (int k = 0; k < kDepth; ++k) see4(v[k], lo + ((k0 + k) * kThreads + tid) * 4);
    }
  } else if (kVec4) {
    // the row's last chunk: whole float4 words, then the ragged end
    for (int e = lo + tid * 4; e < hi; e += kThreads * 4) {
      if (e + 4 <= hi) {
        see4(__ldcs(reinterpret_cast<const float4 *>(src + e)), e);
      } else {
        for (int q = e; q < hi; ++q) see1(src[q], q);
      }
    }
  } else {
    for (int e = lo + tid; e < hi; e += kThreads) see1(src[e], e);
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

namespace {

// The row argmax of logits (or of the rows' sampled scores when sp.N > 0).
int row_argmax(const float *logits, int64_t rows, int vocab, int64_t row_stride, int32_t *argmax, void *workspace,
               size_t ws_bytes, const Sampler &sp, cudaStream_t s) {
  if (rows < 0 || vocab < 1 || row_stride < vocab) return DTS_ERR_INVALID;
  if (rows == 0) return DTS_OK;
  if (!logits || !argmax || (reinterpret_cast<uintptr_t>(logits) & 3)) return DTS_ERR_INVALID;
  const int chunks = chunks_of(vocab);
  if (rows * chunks >= (1ll << 31)) return DTS_ERR_UNSUPPORTED;
  if (workspace == nullptr || ws_bytes < dts_target_argmax_workspace(rows, vocab)) return DTS_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 7) return DTS_ERR_INVALID;
  uint64_t *best = static_cast<uint64_t *>(workspace);
  const unsigned blocks = static_cast<unsigned>(rows * chunks);
  const bool vec4 = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && (row_stride & 3) == 0;
  const bool sample = sp.N > 0;
  if (vec4 && sample) argmax_chunk_kernel<true, true><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best, sp);
  else if (vec4) argmax_chunk_kernel<true, false><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best, sp);
  else if (sample) argmax_chunk_kernel<false, true><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best, sp);
  else argmax_chunk_kernel<false, false><<<blocks, kThreads, 0, s>>>(logits, row_stride, vocab, chunks, best, sp);
  if (dts_host::launch_status() != DTS_OK) return DTS_ERR_CUDA;
  argmax_reduce_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(best, rows, chunks, argmax);
  return dts_host::launch_status();
}

}  // namespace

extern "C" int dts_target_argmax(const float *logits, int64_t rows, int vocab, int64_t row_stride, int32_t *argmax,
                                 void *workspace, size_t ws_bytes, dts_stream_t stream) {
  return row_argmax(logits, rows, vocab, row_stride, argmax, workspace, ws_bytes, Sampler{nullptr, nullptr, nullptr, nullptr, 0},
                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dts_sample_draws(const float *logits, int vocab, int64_t row_stride, const int32_t *vc,
                                const int32_t *depth, const float *temperature, const uint64_t *seed, int B, int N,
                                int32_t *draws, void *workspace, size_t ws_bytes, dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (B == 0) return DTS_OK;
  if (!vc || !depth || !temperature || !seed) return DTS_ERR_INVALID;
  return row_argmax(logits, static_cast<int64_t>(B) * N, vocab, row_stride, draws, workspace, ws_bytes,
                    Sampler{vc, depth, temperature, seed, N}, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int dts_verify_tree_sampled(const int32_t *draft_tokens, const float *logits, int vocab, int64_t row_stride,
                                       const int32_t *vc, const int32_t *depth, const float *temperature,
                                       const uint64_t *seed, const int32_t *parents, const int32_t *next_token,
                                       const int32_t *next_sibling, int B, int N, int32_t *draws,
                                       int32_t *accept_len, int32_t *accepted_path, int32_t *accepted_tokens,
                                       void *workspace, size_t ws_bytes, int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes) return DTS_ERR_UNSUPPORTED;
  if (B == 0) return DTS_OK;
  if (!draft_tokens || !draws || !accept_len || !accepted_path || !accepted_tokens) return DTS_ERR_INVALID;
  if ((next_token == nullptr) != (next_sibling == nullptr)) return DTS_ERR_INVALID;
  if (next_token == nullptr && parents == nullptr) return DTS_ERR_INVALID;
  const int st = dts_sample_draws(logits, vocab, row_stride, vc, depth, temperature, seed, B, N, draws, workspace,
                                  ws_bytes, stream);
  if (st != DTS_OK) return st;
  return dts_verify_tree_greedy(draft_tokens, draws, parents, next_token, next_sibling, B, N, accept_len,
                                accepted_path, accepted_tokens, err_dev, stream);
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
