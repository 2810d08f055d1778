// Compaction of the accepted path, shared by the compaction kernels and the
// fused verify epilogue: KV rows of every buffer in a cache group's address
// table, and hidden rows plus positions.
//
// [TS] "The tree is a parameter of the chain path": the path's KV of every
// layer moves to the window's leading slots by a word copy that does not care
// about dtype, and the hidden rows move to the front of the window with the
// positions back to vc + i. [MI] "Discarding the rejected branches' KV":
// destinations are the first accept_len window slots.
//
// Snapshot order: the accepted path is strictly increasing with path[0] = 0,
// so path[t] >= t. A row written for step t (window slot t) is never the
// source of a later step t2 > t (whose source is slot path[t2] >= t2 > t).
// The copy therefore runs in rounds over the moved rows in ascending order:
// each round loads all of its words into registers, the block synchronises,
// then stores them. Within a round every load precedes every store; across
// rounds the argument above holds.
#pragma once

#include "common.cuh"

namespace dts {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;  // words staged per thread per round

// Validate one request's packed path with one warp (lane l looks at steps l
// and l + 32; N <= 64). Fills dst/src with the moved rows (in window-slot
// units, ascending) and returns their count in every lane, or -1 for a bad
// path.
__device__ __forceinline__ int collect_moves_warp(const int32_t *path, int alen, int N, int *dst, int *src) {
  const int lane = threadIdx.x & 31;
  if (alen < 1 || alen > N) return -1;
  int n = 0;
  bool bad = false;
  int prev_hi = 0;  // path[31], the predecessor of step 32
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int t = half * 32 + lane;
    const int p = t < alen ? path[t] : 0;
    int before = __shfl_up_sync(0xffffffffu, p, 1);
    if (lane == 0) before = prev_hi;
    prev_hi = __shfl_sync(0xffffffffu, p, 31);
    if (t < alen) {
      if (t == 0) bad |= p != 0;
      else bad |= p <= before || p >= N;
    }
    const bool moves = t >= 1 && t < alen && p != t;
    const uint32_t m = __ballot_sync(0xffffffffu, moves);
    if (moves) {
      const int k = n + __popc(m & ((1u << lane) - 1u));
      dst[k] = t;
      src[k] = p;
    }
    n += __popc(m);
  }
  return __any_sync(0xffffffffu, bad) ? -1 : n;
}

template <typename Word>
__device__ __forceinline__ void move_rows(char *base, int64_t stride, int row_words, const int64_t *dst_slot,
                          const int64_t *src_slot, int n_moved) {
  const int64_t total = static_cast<int64_t>(n_moved) * row_words;
  for (int64_t r0 = 0; r0 < total; r0 += static_cast<int64_t>(kThreads) * kPerThread) {
    Word v[kPerThread];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int64_t e = r0 + static_cast<int64_t>(k) * kThreads + threadIdx.x;
      if (e < total) {
        const int m = static_cast<int>(e / row_words);
        const int c = static_cast<int>(e % row_words);
        v[k] = reinterpret_cast<const Word *>(base + src_slot[m] * stride)[c];
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int64_t e = r0 + static_cast<int64_t>(k) * kThreads + threadIdx.x;
      if (e < total) {
        const int m = static_cast<int>(e / row_words);
        const int c = static_cast<int>(e % row_words);
        reinterpret_cast<Word *>(base + dst_slot[m] * stride)[c] = v[k];
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void move_rows_any(char *base, int64_t stride, int row_bytes, const int64_t *dst_slot,
                              const int64_t *src_slot, int n_moved) {
  const uint64_t a = reinterpret_cast<uint64_t>(base) | static_cast<uint64_t>(stride) |
                     static_cast<uint64_t>(row_bytes);
  if ((a & 15) == 0) move_rows<uint4>(base, stride, row_bytes / 16, dst_slot, src_slot, n_moved);
  else if ((a & 7) == 0) move_rows<uint2>(base, stride, row_bytes / 8, dst_slot, src_slot, n_moved);
  else move_rows<uint32_t>(base, stride, row_bytes / 4, dst_slot, src_slot, n_moved);
}

constexpr int kBufPerBlock = 8;  // buffers of the table one block moves

// Shared state of one block's KV compaction (kv_prepare, then kv_move).
struct KvCompactSmem {
  int dst[kMaxNodes], src[kMaxNodes];        // moved rows, in window-slot units
  int64_t dslot[kMaxNodes], sslot[kMaxNodes];
  int64_t wl[kMaxNodes];                      // the request's window slots
  dts_kv_buffer e[kBufPerBlock];
  int skip[kBufPerBlock];
  int64_t pref[kBufPerBlock + 1];             // words (16-byte) before buffer k's rows
  int n, all16;
};

// The part of request b's KV compaction in buffers [gx * kBufPerBlock, ...)
// of the table that does not need its path: the buffers' entries and their
// checks, the overlap verdicts between entries, and the request's window
// slots. Threads tid = 0 .. nthr - 1 of the block take part, whole warps,
// nthr a multiple of 32 (the rest may be walking the tree meanwhile); they
// meet once on hardware barrier 1. Nothing is reported yet, and the caller
// synchronises the block before kv_move.
__device__ __forceinline__ void kv_prepare(const dts_kv_buffer *__restrict__ table, int n_buffers, int gx,
                                           const int64_t *__restrict__ wl, int b, int N, KvCompactSmem &s, int tid,
                                           int nthr) {
  const int l0 = gx * kBufPerBlock;
  const int nb = min(kBufPerBlock, n_buffers - l0);
  for (int k = tid; k < nb; k += nthr) {
    const dts_kv_buffer e = table[l0 + k];
    s.e[k] = e;
    const uint64_t al = reinterpret_cast<uint64_t>(e.base) | static_cast<uint64_t>(e.slot_stride_bytes) |
                        static_cast<uint64_t>(e.row_bytes);
    const bool bad = e.base == nullptr || (al & 3) != 0 || e.row_bytes <= 0 || e.slot_stride_bytes < e.row_bytes ||
                     e.num_slots <= 0 || e.reserved != 0;
    s.skip[k] = bad ? 1 : 0;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory");
  // Each physical region moves once: skip an entry if another entry with the
  // same stride covers its rows (equal ranges: the lower index moves).
  for (int q = tid; q < nb * n_buffers; q += nthr) {
    const int k = q / n_buffers, o = q - k * n_buffers;
    const int l = l0 + k;
    if (o == l || s.skip[k] == 1) continue;
    const dts_kv_buffer e = s.e[k];
    const dts_kv_buffer f = table[o];
    if (f.slot_stride_bytes != e.slot_stride_bytes || f.base == nullptr) continue;
    const uint64_t lo = reinterpret_cast<uint64_t>(e.base);
    const uint64_t hi = lo + static_cast<uint64_t>(e.row_bytes);
    const uint64_t flo = reinterpret_cast<uint64_t>(f.base);
    const uint64_t fhi = flo + static_cast<uint64_t>(f.row_bytes);
    if (fhi <= lo || hi <= flo) continue;                     // disjoint
    const bool inside = flo <= lo && hi <= fhi;
    const bool outside = lo <= flo && fhi <= hi;
    if (inside && !(outside && o > l)) atomicOr(&s.skip[k], 2);  // covered by o
    else if (!inside && !outside) atomicOr(&s.skip[k], 4);       // partial overlap
  }
  for (int j = tid; j < N; j += nthr) s.wl[j] = wl[static_cast<int64_t>(b) * N + j];
}

// The rest, once kv_prepare's writes are visible to the block: request b's
// path rows move in the prepared buffers. `path` points at the request's
// packed path (global or shared memory), `alen` is its length. When every
// buffer is 16-byte aligned, all their moved rows go in one load-then-store
// round. Errors are reported in the order the checks are defined: a bad
// entry, a bad path, a partial overlap, a slot out of range.
__device__ __forceinline__ void kv_move(int n_buffers, int gx, const int32_t *path, int alen, int b, int N,
                                        KvCompactSmem &s, int32_t *err) {
  const int nb = min(kBufPerBlock, n_buffers - gx * kBufPerBlock);
  if (threadIdx.x < nb && s.skip[threadIdx.x] == 1) report(err, DTS_DEV_BAD_BUFFER);
  __syncthreads();
  if (threadIdx.x < 32) {
    const int n = collect_moves_warp(path, alen, N, s.dst, s.src);
    __syncwarp();
    if (n < 0) {
      if (threadIdx.x == 0) {
        if (gx == 0) report(err, DTS_DEV_BAD_PATH);
        s.n = 0;
      }
    } else {
      for (int m = threadIdx.x; m < n; m += 32) {
        s.dslot[m] = s.wl[s.dst[m]];
        s.sslot[m] = s.wl[s.src[m]];
      }
      if (threadIdx.x == 0) s.n = n;
    }
  }
  __syncthreads();
  const int n_moved = s.n;
  if (n_moved == 0) return;
  if (threadIdx.x < nb) {
    // slots in range for this buffer, the overlap verdicts, 16-byte words
    const dts_kv_buffer e = s.e[threadIdx.x];
    int skip = s.skip[threadIdx.x];
    if (skip & 4) {
      if (b == 0) report(err, DTS_DEV_BAD_BUFFER);
    }
    if (skip == 0) {
      bool bad = false;
      for (int m = 0; m < n_moved; ++m)
        bad |= s.dslot[m] < 0 || s.dslot[m] >= e.num_slots || s.sslot[m] < 0 || s.sslot[m] >= e.num_slots;
      if (bad) {
        report(err, DTS_DEV_BAD_SLOT);
        skip = 8;
      }
    }
    s.skip[threadIdx.x] = skip;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t acc = 0;
    int all16 = 1;
    for (int k = 0; k < nb; ++k) {
      s.pref[k] = acc;
      if (s.skip[k] != 0) continue;
      const dts_kv_buffer e = s.e[k];
      const uint64_t al = reinterpret_cast<uint64_t>(e.base) | static_cast<uint64_t>(e.slot_stride_bytes) |
                          static_cast<uint64_t>(e.row_bytes);
      all16 &= (al & 15) == 0 ? 1 : 0;
      acc += static_cast<int64_t>(n_moved) * (e.row_bytes / 16);
    }
    s.pref[nb] = acc;
    s.all16 = all16;
  }
  __syncthreads();
  if (!s.all16) {
    for (int k = 0; k < nb; ++k)
      if (s.skip[k] == 0)
        move_rows_any(static_cast<char *>(s.e[k].base), s.e[k].slot_stride_bytes, s.e[k].row_bytes, s.dslot,
                      s.sslot, n_moved);
    return;
  }
  // every moved row of every buffer, as 16-byte words, in rounds
  const int64_t total = s.pref[nb];
  for (int64_t r0 = 0; r0 < total; r0 += static_cast<int64_t>(kThreads) * kPerThread) {
    uint4 v[kPerThread];
    char *dst_addr[kPerThread];
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      const int64_t e = r0 + static_cast<int64_t>(q) * kThreads + threadIdx.x;
      dst_addr[q] = nullptr;
      if (e < total) {
        int k = 0;
        while (k + 1 < nb && s.pref[k + 1] <= e) ++k;
        const int64_t row_words = s.e[k].row_bytes / 16;
        const int64_t local = e - s.pref[k];
        const int m = static_cast<int>(local / row_words);
        const int64_t c = local - m * row_words;
        char *base = static_cast<char *>(s.e[k].base);
        v[q] = reinterpret_cast<const uint4 *>(base + s.sslot[m] * s.e[k].slot_stride_bytes)[c];
        dst_addr[q] = base + s.dslot[m] * s.e[k].slot_stride_bytes + c * 16;
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPerThread; ++q)
      if (dst_addr[q] != nullptr) *reinterpret_cast<uint4 *>(dst_addr[q]) = v[q];
    __syncthreads();
  }
}

// Request b's positions back to vc + i (threads tid = 0 .. nthr - 1).
__device__ __forceinline__ void write_positions(int32_t *__restrict__ positions, const int32_t *__restrict__ vc,
                                                int b, int N, int tid, int nthr) {
  if (positions == nullptr) return;
  const int v = vc[b];
  for (int i = tid; i < N; i += nthr) positions[static_cast<int64_t>(b) * N + i] = v + i;
}

// One block: request b's hidden rows along its path (global or shared
// `path`, length `alen`).
__device__ __forceinline__ void move_hidden_block(char *__restrict__ hidden, int64_t row_bytes, const int32_t *path,
                                                  int alen, int b, int N, int32_t *err) {
  __shared__ int s_dst[kMaxNodes], s_src[kMaxNodes];
  __shared__ int64_t s_dslot[kMaxNodes], s_sslot[kMaxNodes];
  __shared__ int s_n;
  if (hidden == nullptr) return;
  if (threadIdx.x < 32) {
    const int n = collect_moves_warp(path, alen, N, s_dst, s_src);
    __syncwarp();
    if (n < 0 && threadIdx.x == 0) report(err, DTS_DEV_BAD_PATH);
    for (int m = threadIdx.x; m < n; m += 32) {
      s_dslot[m] = static_cast<int64_t>(b) * N + s_dst[m];
      s_sslot[m] = static_cast<int64_t>(b) * N + s_src[m];
    }
    if (threadIdx.x == 0) s_n = n < 0 ? 0 : n;
  }
  __syncthreads();
  if (s_n == 0) return;
  move_rows_any(hidden, row_bytes, static_cast<int>(row_bytes), s_dslot, s_sslot, s_n);
}

}  // namespace dts
