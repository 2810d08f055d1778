// Tree-verify attention: every verify row attends the committed prefix plus
// its own ancestors in the window.
//
// [TS] "One tree attention": every row sees the committed prefix, and the
// 64-bit ancestor mask applies only to the window keys; the prefix is where
// the time goes at long context; results carry a base-2 log-sum-exp.
// [AK] section one: row v equals Target(prefix + path(root -> v)).
// [AK] section four: partial results over disjoint key sets merge by their
// log-sum-exps, O = sum Z_k O_k / sum Z_k.
//
// Two kernels:
//
// 1. prefix pass (tcgen05): one CTA per (request, KV head, 256-row pair, KV
//    split). The rows of a KV head are the N*g (node, query head) pairs, so a
//    CTA holds up to two 128-row tiles and reads each K/V page once for all of
//    them. TMA brings 128-key K and V tiles (128-byte swizzle, one box per
//    page and 64-column block) into a ring of shared-memory slots; one thread
//    issues S = Q K^T into tensor memory; each 128-thread softmax group owns
//    one row tile (thread = TMEM lane = row), turns S into bf16 P in place
//    (P aliases the first half of S's columns) and the MMA thread issues
//    O += P V with P read straight from TMEM. The running max is rescaled
//    lazily (only when it grows by more than 2^8), so O is rarely touched.
//    Output: normalised fp32 partial O and its base-2 LSE per split.
//
// 2. window + merge pass (SIMT): one warp per (node, KV head, head group).
//    It merges the prefix splits by their LSEs, then walks the set bits of
//    the node's ancestor mask (only those window keys are ever read, so
//    non-finite values in unseen slots cannot leak), and writes bf16 out and
//    the fp32 base-2 LSE.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace {

using namespace dts::ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPlanTargetCtas = 4 * 152;  // a few waves of GB300's 152 SMs
constexpr int kMinChunk = 512;

struct Plan {
  int n_pairs, n_splits, chunk;
  int64_t o_bytes, lse_bytes;
};

Plan make_plan(int B, int N, int Hq, int Hkv, int d, int64_t max_prefix) {
  Plan p;
  const int g = Hq / Hkv;
  const int M = N * g;
  p.n_pairs = (M + 255) / 256;
  const int64_t units = static_cast<int64_t>(B) * Hkv * p.n_pairs;
  int64_t want = (kPlanTargetCtas + units - 1) / units;
  const int64_t max_splits = max_prefix > 0 ? (max_prefix + kMinChunk - 1) / kMinChunk : 1;
  if (want > max_splits) want = max_splits;
  if (want < 1) want = 1;
  int64_t c = max_prefix > 0 ? (max_prefix + want - 1) / want : 128;
  c = ((c + 127) / 128) * 128;
  if (c < 128) c = 128;
  p.chunk = static_cast<int>(c);
  p.n_splits = max_prefix > 0 ? static_cast<int>((max_prefix + c - 1) / c) : 1;
  const int64_t rows = static_cast<int64_t>(B) * N * Hq;
  p.o_bytes = static_cast<int64_t>(p.n_splits) * rows * d * 4;
  p.lse_bytes = static_cast<int64_t>(p.n_splits) * rows * 4;
  return p;
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// ============================================================================
// prefix pass
// ============================================================================
struct PrefixArgs {
  const uint16_t *q;
  const int32_t *page_table;
  const int32_t *prefix_len;
  const int32_t *positions;
  float *o_part;
  float *lse_part;
  int32_t *err;
  int64_t num_slots, max_prefix;
  int B, N, Hq, Hkv, g, M, n_pairs, n_splits, chunk, max_pages, page_shift;
  float scale_log2;
  dts::RopeFreqs freqs;
};

template <int D>
struct PrefixShape {
  static constexpr int kThreads = 384;              // 4 control warps + 2 softmax groups
  static constexpr uint32_t kTileBytes = 128 * D * 2;  // a 128-row bf16 tile (Q, K or V)
  static constexpr uint32_t kBlockBytes = 128 * 128;   // one 64-column block of a 128-row tile
  static constexpr int kSlots = D == 128 ? 5 : 8;      // K/V ring
  static constexpr uint32_t kBarBytes = 256;
  static constexpr uint32_t kSmem = 1024 /*align*/ + 2 * kTileBytes + kSlots * kTileBytes + kBarBytes;
};

// Shared-memory position of element `e` of row `r` in a K-major tile with
// 128-byte swizzle: 64-column blocks of 128 rows x 128 B; 16-byte chunk c of
// row r sits at chunk c ^ (r & 7).
__device__ __forceinline__ uint32_t sw128_offset(int r, int e) {
  const int cb = e >> 6;
  const int ch = (e & 63) >> 3;
  return static_cast<uint32_t>(cb * (128 * 128) + r * 128 + ((ch ^ (r & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void load_q_tiles(const PrefixArgs &a, uint8_t *sQ, int b, int hkv, int row0, int nt) {
  constexpr int kPairChunks = D / 16;  // 8-element chunks in the first half of a row
  constexpr uint32_t kTileBytes = PrefixShape<D>::kTileBytes;
  const int items = nt * 128 * kPairChunks;
  for (int it = threadIdx.x; it < items; it += PrefixShape<D>::kThreads) {
    const int c = it % kPairChunks;
    const int rr = it / kPairChunks;
    const int t = rr >> 7;
    const int r = rr & 127;
    const int R = row0 + t * 128 + r;
    uint4 x1 = make_uint4(0, 0, 0, 0), x2 = make_uint4(0, 0, 0, 0);
    if (R < a.M) {
      const int i = R / a.g;
      const int hh = R - i * a.g;
      const int64_t node = static_cast<int64_t>(b) * a.N + i;
      const uint16_t *src = a.q + (node * a.Hq + static_cast<int64_t>(hkv) * a.g + hh) * D;
      x1 = *reinterpret_cast<const uint4 *>(src + 8 * c);
      x2 = *reinterpret_cast<const uint4 *>(src + D / 2 + 8 * c);
      if (a.positions != nullptr) {
        const int pos = a.positions[node];
        uint32_t *w1 = reinterpret_cast<uint32_t *>(&x1);
        uint32_t *w2 = reinterpret_cast<uint32_t *>(&x2);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float s0, c0, s1, c1;
          dts::rope_sincos(pos, a.freqs.w[8 * c + 2 * e], &s0, &c0);
          dts::rope_sincos(pos, a.freqs.w[8 * c + 2 * e + 1], &s1, &c1);
          const float u0 = dts::bf16_lo(w1[e]), u1 = dts::bf16_hi(w1[e]);
          const float v0 = dts::bf16_lo(w2[e]), v1 = dts::bf16_hi(w2[e]);
          w1[e] = dts::pack_bf16x2(u0 * c0 - v0 * s0, u1 * c1 - v1 * s1);
          w2[e] = dts::pack_bf16x2(v0 * c0 + u0 * s0, v1 * c1 + u1 * s1);
        }
      }
    }
    uint8_t *tile = sQ + t * kTileBytes;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 8 * c)) = x1;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, D / 2 + 8 * c)) = x2;
  }
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    tree_prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ PrefixArgs a) {
  using S = PrefixShape<D>;
  constexpr int kSlots = S::kSlots;
  constexpr uint32_t kTileBytes = S::kTileBytes;
  constexpr int kKSteps = D / 16;  // K-steps of S = Q K^T
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: (request, KV head, KV split, row pair) ----
  int idx = blockIdx.x;
  const int pair = idx % a.n_pairs;
  idx /= a.n_pairs;
  const int split = idx % a.n_splits;
  idx /= a.n_splits;
  const int hkv = idx % a.Hkv;
  const int b = idx / a.Hkv;
  const int P = a.prefix_len[b];
  if (P < 0 || P > a.max_prefix ||
      static_cast<int64_t>(P) + a.N > (static_cast<int64_t>(a.max_pages) << a.page_shift))
    return;  // reported by the window pass
  const int lo = split * a.chunk;
  if (lo >= P) return;
  const int hi = min(P, lo + a.chunk);
  const int nkt = (hi - lo + 127) >> 7;
  const int row0 = pair * 256;
  const int nt = min(2, (a.M - row0 + 127) >> 7);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sQ = smem;
  uint8_t *sKV = smem + 2 * kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sKV + kSlots * kTileBytes);
  uint64_t *full = bars;
  uint64_t *empty = bars + kSlots;
  uint64_t *s_full = bars + 2 * kSlots;
  uint64_t *p_full = s_full + 2;
  uint64_t *o_fin = p_full + 2;
  uint64_t *drain = o_fin + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_fin[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  load_q_tiles<D>(a, sQ, b, hkv, row0, nt);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ_addr = smem_addr(sQ);
  const uint32_t sKV_addr = smem_addr(sKV);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int ps = 1 << a.page_shift;
      const int rows_per_box = ps < 128 ? ps : 128;
      const int boxes = 128 / rows_per_box;
      const int64_t pt_row = static_cast<int64_t>(b) * a.max_pages;
      int use = 0;
      bool ok = true;
      for (int j = 0; j < nkt && ok; ++j) {
        const int kbase = lo + j * 128;
        const int nvalid = min(128, hi - kbase);
        for (int kv = 0; kv < 2 && ok; ++kv, ++use) {
          const int slot = use % kSlots;
          const uint32_t ph = static_cast<uint32_t>(use / kSlots) & 1u;
          if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag)) {
            dts::report(a.err, DTS_DEV_TIMEOUT);
            ok = false;
            break;
          }
          // count the boxes first: the barrier must expect exactly their bytes
          int nbox = 0;
          int coord[16];
          for (int r = 0; r < boxes; ++r) {
            coord[r] = -1;
            const int key = kbase + r * rows_per_box;
            if (r * rows_per_box >= nvalid) continue;
            const int pid = a.page_table[pt_row + (key >> a.page_shift)];
            const int64_t s0 = static_cast<int64_t>(pid) * ps + (key & (ps - 1));
            if (pid < 0 || s0 + rows_per_box > a.num_slots) {
              dts::report(a.err, DTS_DEV_BAD_SLOT);
              continue;
            }
            coord[r] = static_cast<int>(s0);
            ++nbox;
          }
          mbar_expect_tx(&full[slot], static_cast<uint32_t>(nbox * rows_per_box * 128 * (D / 64)));
          const CUtensorMap *map = kv == 0 ? &tm_k : &tm_v;
          const uint32_t dst = sKV_addr + slot * kTileBytes;
          for (int r = 0; r < boxes; ++r) {
            if (coord[r] < 0) continue;
            for (int h = 0; h < D / 64; ++h)
              tma_load_3d(dst + h * S::kBlockBytes + r * rows_per_box * 128, map, h * 64, hkv, coord[r],
                          &full[slot]);
          }
        }
      }
      if (!ok) {
        // give the copies already in flight a bounded chance to land
        for (int u = max(0, use - kSlots); u < use; ++u)
          mbar_wait(&full[u % kSlots], static_cast<uint32_t>(u / kSlots) & 1u, abort_flag);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
    constexpr uint32_t kIdescO = idesc_bf16(128, D, true);
    bool ok = true;
    auto slot_of = [](int use) { return use % kSlots; };
    auto phase_of = [](int use) { return static_cast<uint32_t>(use / kSlots) & 1u; };
    auto issue_s = [&](int t, int slot) {
      const uint32_t qa = sQ_addr + t * kTileBytes;
      const uint32_t kb = sKV_addr + slot * kTileBytes;
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        const uint32_t off = (ks >> 2) * S::kBlockBytes + (ks & 3) * 32;
        mma_ss(tmem + t * 256, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), kIdescS,
               ks > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int slot, bool first) {
      const uint32_t vb = sKV_addr + slot * kTileBytes;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // 128 keys, 16 per step
        mma_ts(tmem + t * 256 + 128, tmem + t * 256 + ks * 8, sdesc_sw128(vb + ks * 2048, S::kBlockBytes, 1024),
               kIdescO, (first && ks == 0) ? 0u : 1u);
      }
    };
    // prologue: S(0)
    if (!mbar_wait(&full[slot_of(0)], phase_of(0), abort_flag)) ok = false;
    tc_fence_after();
    if (ok && lane == 0) {
      for (int t = 0; t < nt; ++t) {
        issue_s(t, slot_of(0));
        mma_commit(&s_full[t]);
      }
      mma_commit(&empty[slot_of(0)]);
    }
    __syncwarp();
    for (int j = 0; j < nkt && ok; ++j) {
      const int vuse = 2 * j + 1;
      const int vslot = slot_of(vuse);
      if (!mbar_wait(&full[vslot], phase_of(vuse), abort_flag)) {
        ok = false;
        break;
      }
      const int nvalid = min(128, hi - (lo + j * 128));
      if (nvalid < 128) {
        // keys past the split's end: zero their V rows so that 0 * (stale or
        // non-finite V) cannot reach O
        uint8_t *vt = sKV + vslot * kTileBytes;
        for (int h = 0; h < D / 64; ++h) {
          uint4 *p = reinterpret_cast<uint4 *>(vt + h * S::kBlockBytes + nvalid * 128);
          const int n16 = (128 - nvalid) * 8;
          for (int e = lane; e < n16; e += 32) p[e] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
        __syncwarp();
      }
      for (int t = 0; t < nt && ok; ++t) {
        if (!mbar_wait(&p_full[t], static_cast<uint32_t>(j) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          issue_pv(t, vslot, j == 0);
          if (t == nt - 1) mma_commit(&empty[vslot]);
          if (j == nkt - 1) mma_commit(&o_fin[t]);
        }
        __syncwarp();
        if (j + 1 < nkt) {
          const int kuse = 2 * (j + 1);
          if (t == 0) {
            if (!mbar_wait(&full[slot_of(kuse)], phase_of(kuse), abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (lane == 0) {
            issue_s(t, slot_of(kuse));
            mma_commit(&s_full[t]);
            if (t == nt - 1) mma_commit(&empty[slot_of(kuse)]);
          }
          __syncwarp();
        }
      }
    }
    if (!ok) dts::report(a.err, DTS_DEV_TIMEOUT);
    // drain: wait for every MMA issued so far before TMEM is released
    if (lane == 0) mma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, abort_flag);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    if (t < nt) {
      const int r = wq * 32 + lane;
      const int R = row0 + t * 128 + r;
      const bool warp_valid = row0 + t * 128 + wq * 32 < a.M;
      const uint32_t tS = tmem + (static_cast<uint32_t>(wq * 32) << 16) + t * 256;
      const uint32_t tO = tS + 128;
      const float c = a.scale_log2;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nkt; ++j) {
        if (!mbar_wait(&s_full[t], static_cast<uint32_t>(j) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp_valid) {
          uint32_t sv[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sv[q]);
          tmem_wait_ld();
          const int nvalid = min(128, hi - (lo + j * 128));
          float mx = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (q * 32 + k < nvalid) mx = fmaxf(mx, __uint_as_float(sv[q][k]));
          const float m_new = mx * c;
          float m_use = m_run;
          if (m_new > m_run + 8.f) m_use = m_new;  // lazy rescale: P stays below 2^8
          const float alpha = ex2(m_run - m_use);
          // P = 2^(s*c - m_use) as bf16 pairs, packed in place over the consumed
          // S registers: pair (q, k) lands in sv[q >> 1][(q & 1) * 16 + k / 2],
          // an entry already read.
          float lsum = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const int col = q * 32 + k;
              const float p0 = col < nvalid ? ex2(fmaf(__uint_as_float(sv[q][k]), c, -m_use)) : 0.f;
              const float p1 = col + 1 < nvalid ? ex2(fmaf(__uint_as_float(sv[q][k + 1]), c, -m_use)) : 0.f;
              lsum += p0 + p1;
              sv[q >> 1][(q & 1) * 16 + (k >> 1)] = dts::pack_bf16x2(p0, p1);
            }
          l_run = l_run * alpha + lsum;
          m_run = m_use;
          tmem_st32(tS, sv[0]);
          tmem_st32(tS + 32, sv[1]);
          // O was last written by PV(j-1), complete before S(j) was: rescale it
          // now if this warp's running max moved.
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int q = 0; q < D / 32; ++q) {
              uint32_t ov[32];
              tmem_ld32(tO + q * 32, ov);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
              tmem_st32(tO + q * 32, ov);
            }
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&p_full[t]);
      }
      if (ok && mbar_wait(&o_fin[t], 0, abort_flag)) {
        tc_fence_after();
        if (warp_valid) {
          const bool valid = R < a.M;
          const int i = R / a.g;
          const int hh = R - i * a.g;
          const int64_t rows = static_cast<int64_t>(a.B) * a.N * a.Hq;
          const int64_t gr = (static_cast<int64_t>(b) * a.N + i) * a.Hq + static_cast<int64_t>(hkv) * a.g + hh;
          const float inv_l = 1.f / l_run;
          float *dst = a.o_part + (static_cast<int64_t>(split) * rows + gr) * D;
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(tO + q * 32, ov);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
              for (int k = 0; k < 32; k += 4) {
                float4 v = make_float4(__uint_as_float(ov[k]) * inv_l, __uint_as_float(ov[k + 1]) * inv_l,
                                       __uint_as_float(ov[k + 2]) * inv_l, __uint_as_float(ov[k + 3]) * inv_l);
                *reinterpret_cast<float4 *>(dst + q * 32 + k) = v;
              }
            }
          }
          if (valid) a.lse_part[static_cast<int64_t>(split) * rows + gr] = m_run + __log2f(l_run);
        }
      } else {
        dts::report(a.err, DTS_DEV_TIMEOUT);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================
// window + merge pass
// ============================================================================
struct WindowArgs {
  const uint16_t *q;
  const uint16_t *k_cache;
  const uint16_t *v_cache;
  const int32_t *page_table;
  const int32_t *prefix_len;
  const uint64_t *mask;
  const int32_t *positions;
  const float *o_part;
  const float *lse_part;
  uint16_t *out;
  float *lse2;
  int32_t *err;
  int64_t num_slots, max_prefix;
  int B, N, Hq, Hkv, g, heads_per_warp, max_pages, page_shift, n_splits, chunk;
  float scale_log2;
  dts::RopeFreqs freqs;
};

// Lane l holds elements {2l, 2l+1, D/2+2l, D/2+2l+1} (D = 128) or {l, D/2+l}
// (D = 64): both halves of its rotate-half pairs.
template <int D>
struct LaneElems {
  static constexpr int kE = D / 32;
};

template <int D>
__device__ __forceinline__ void load_row(const uint16_t *row, int lane, float (&x)[D / 32]) {
  if constexpr (D == 128) {
    const uint32_t w1 = reinterpret_cast<const uint32_t *>(row)[lane];
    const uint32_t w2 = reinterpret_cast<const uint32_t *>(row + 64)[lane];
    x[0] = dts::bf16_lo(w1);
    x[1] = dts::bf16_hi(w1);
    x[2] = dts::bf16_lo(w2);
    x[3] = dts::bf16_hi(w2);
  } else {
    x[0] = __uint_as_float(static_cast<uint32_t>(row[lane]) << 16);
    x[1] = __uint_as_float(static_cast<uint32_t>(row[32 + lane]) << 16);
  }
}

template <int D>
__device__ __forceinline__ int elem_index(int lane, int e) {
  if constexpr (D == 128) return (e < 2) ? 2 * lane + e : 64 + 2 * lane + (e - 2);
  else return e == 0 ? lane : 32 + lane;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int D, int HW>
__global__ void __launch_bounds__(256) tree_window_kernel(const __grid_constant__ WindowArgs a) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int groups = a.g / HW;
  const int64_t total = static_cast<int64_t>(a.B) * a.N * a.Hkv * groups;
  if (wid >= total) return;
  const int hg = static_cast<int>(wid % groups);
  wid /= groups;
  const int hkv = static_cast<int>(wid % a.Hkv);
  const int64_t node = wid / a.Hkv;  // b * N + i
  const int b = static_cast<int>(node / a.N);
  const int h0 = hkv * a.g + hg * HW;
  const int P = a.prefix_len[b];
  const int64_t rows = static_cast<int64_t>(a.B) * a.N * a.Hq;

  if (P < 0 || P > a.max_prefix ||
      static_cast<int64_t>(P) + a.N > (static_cast<int64_t>(a.max_pages) << a.page_shift)) {
    if (lane == 0) dts::report(a.err, DTS_DEV_BAD_SLOT);
    for (int u = 0; u < HW; ++u) {
      uint16_t *o = a.out + (node * a.Hq + h0 + u) * D;
      for (int e = lane; e < D; e += 32) o[e] = 0x7FC0;  // NaN
      if (lane == 0) a.lse2[node * a.Hq + h0 + u] = __int_as_float(0x7FC00000);
    }
    return;
  }

  // queries, rotated (fp32) and held in the model dtype
  float q[HW][E];
  const int pos = a.positions != nullptr ? a.positions[node] : 0;
#pragma unroll
  for (int u = 0; u < HW; ++u) {
    load_row<D>(a.q + (node * a.Hq + h0 + u) * D, lane, q[u]);
    if (a.positions != nullptr) {
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const int k = elem_index<D>(lane, e);
        float s, c;
        dts::rope_sincos(pos, a.freqs.w[k], &s, &c);
        const float x1 = q[u][e], x2 = q[u][e + E / 2];
        // the rotated query in the model dtype (bf16), as the prefix pass's MMA sees it
        const uint32_t r = dts::pack_bf16x2(x1 * c - x2 * s, x2 * c + x1 * s);
        q[u][e] = dts::bf16_lo(r);
        q[u][e + E / 2] = dts::bf16_hi(r);
      }
    }
  }

  float m[HW], l[HW], acc[HW][E];
#pragma unroll
  for (int u = 0; u < HW; ++u) {
    m[u] = -INFINITY;
    l[u] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[u][e] = 0.f;
  }

  // prefix partials
  for (int s = 0; s < a.n_splits; ++s) {
    if (s * a.chunk >= P) break;
#pragma unroll
    for (int u = 0; u < HW; ++u) {
      const int64_t gr = static_cast<int64_t>(s) * rows + node * a.Hq + h0 + u;
      const float ls = a.lse_part[gr];
      const float *op = a.o_part + gr * D;
      const float mn = fmaxf(m[u], ls);
      const float sa = dts::ptx::ex2(m[u] - mn), sb = dts::ptx::ex2(ls - mn);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[u][e] = acc[u][e] * sa + op[elem_index<D>(lane, e)] * sb;
      l[u] = l[u] * sa + sb;
      m[u] = mn;
    }
  }

  // window: the node's ancestors (and itself), in ascending node index
  const int ps = 1 << a.page_shift;
  uint64_t mk = a.mask[node];
  if (a.N < 64) mk &= (1ull << a.N) - 1;
  const int64_t pt_row = static_cast<int64_t>(b) * a.max_pages;
  while (mk) {
    const int j = __ffsll(static_cast<long long>(mk)) - 1;
    mk &= mk - 1;
    const int64_t logical = static_cast<int64_t>(P) + j;
    const int pid = a.page_table[pt_row + (logical >> a.page_shift)];
    const int64_t slot = static_cast<int64_t>(pid) * ps + (logical & (ps - 1));
    if (pid < 0 || slot >= a.num_slots) {
      if (lane == 0) dts::report(a.err, DTS_DEV_BAD_SLOT);
      continue;
    }
    float kx[E], vx[E];
    load_row<D>(a.k_cache + (slot * a.Hkv + hkv) * D, lane, kx);
    load_row<D>(a.v_cache + (slot * a.Hkv + hkv) * D, lane, vx);
#pragma unroll
    for (int u = 0; u < HW; ++u) {
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(q[u][e], kx[e], d);
      const float s2 = warp_sum(d) * a.scale_log2;
      const float mn = fmaxf(m[u], s2);
      const float sa = dts::ptx::ex2(m[u] - mn), sb = dts::ptx::ex2(s2 - mn);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[u][e] = acc[u][e] * sa + vx[e] * sb;
      l[u] = l[u] * sa + sb;
      m[u] = mn;
    }
  }

#pragma unroll
  for (int u = 0; u < HW; ++u) {
    const float inv = l[u] > 0.f ? 1.f / l[u] : 0.f;
    uint16_t *o = a.out + (node * a.Hq + h0 + u) * D;
    if constexpr (D == 128) {
      reinterpret_cast<uint32_t *>(o)[lane] = dts::pack_bf16x2(acc[u][0] * inv, acc[u][1] * inv);
      reinterpret_cast<uint32_t *>(o + 64)[lane] = dts::pack_bf16x2(acc[u][2] * inv, acc[u][3] * inv);
    } else {
      const uint32_t w = dts::pack_bf16x2(acc[u][0] * inv, acc[u][1] * inv);
      o[lane] = static_cast<uint16_t>(w & 0xFFFFu);
      o[32 + lane] = static_cast<uint16_t>(w >> 16);
    }
    if (lane == 0) a.lse2[node * a.Hq + h0 + u] = l[u] > 0.f ? m[u] + __log2f(l[u]) : -INFINITY;
  }
}

// ============================================================================
// host side
// ============================================================================
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D view (d, Hkv, slots) of a paged bf16 cache; box (64, 1, rows_per_box).
bool make_cache_map(CUtensorMap *map, const void *base, int d, int Hkv, int64_t num_slots, int rows_per_box) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(num_slots)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(rows_per_box)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
int launch_prefix(const CUtensorMap &tk, const CUtensorMap &tv, const PrefixArgs &a, int grid, cudaStream_t s) {
  using S = PrefixShape<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(tree_prefix_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(S::kSmem));
  });
  if (attr_err != cudaSuccess) return DTS_ERR_CUDA;
  tree_prefix_kernel<D><<<grid, S::kThreads, S::kSmem, s>>>(tk, tv, a);
  return dts_host::launch_status();
}

template <int D>
int launch_window(const WindowArgs &a, cudaStream_t s) {
  const int64_t warps = static_cast<int64_t>(a.B) * a.N * a.Hkv * (a.g / a.heads_per_warp);
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  switch (a.heads_per_warp) {
    case 1: tree_window_kernel<D, 1><<<blocks, 256, 0, s>>>(a); break;
    case 2: tree_window_kernel<D, 2><<<blocks, 256, 0, s>>>(a); break;
    case 4: tree_window_kernel<D, 4><<<blocks, 256, 0, s>>>(a); break;
    default: tree_window_kernel<D, 8><<<blocks, 256, 0, s>>>(a); break;
  }
  return dts_host::launch_status();
}

}  // namespace

extern "C" size_t dts_tree_verify_attention_workspace(int B, int N, int Hq, int Hkv, int d, int64_t max_prefix) {
  if (B <= 0 || N < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || (d != 64 && d != 128) || max_prefix < 0)
    return 0;
  const Plan p = make_plan(B, N, Hq, Hkv, d, max_prefix);
  return static_cast<size_t>(align_up(p.o_bytes, 256) + align_up(p.lse_bytes, 256));
}

extern "C" int dts_tree_verify_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                         int64_t num_slots, const int32_t *page_table, int max_pages,
                                         int page_size, const int32_t *prefix_len, int64_t max_prefix,
                                         const uint64_t *mask, const int32_t *positions, float rope_theta,
                                         int B, int N, int Hq, int Hkv, int d, float softmax_scale,
                                         uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                         int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1 || Hkv < 1 || Hq < 1 || max_pages < 1 || num_slots < 1 || max_prefix < 0)
    return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes || (d != 64 && d != 128)) return DTS_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return DTS_ERR_INVALID;
  if (page_size < 8 || page_size > 4096 || (page_size & (page_size - 1)) != 0) return DTS_ERR_UNSUPPORTED;
  if (max_prefix > (1ll << 30) || num_slots >= (1ll << 31)) return DTS_ERR_UNSUPPORTED;
  if (positions != nullptr && !(rope_theta > 0.f)) return DTS_ERR_INVALID;
  if (B == 0) return DTS_OK;
  if (!q || !k_cache || !v_cache || !page_table || !prefix_len || !mask || !out || !lse2) return DTS_ERR_INVALID;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out) |
                       reinterpret_cast<uintptr_t>(workspace);
  if (al & 15) return DTS_ERR_INVALID;
  const int g = Hq / Hkv;
  if (static_cast<int64_t>(B) * N * Hq >= (1ll << 31) / d) return DTS_ERR_UNSUPPORTED;
  const Plan plan = make_plan(B, N, Hq, Hkv, d, max_prefix);
  const size_t need = dts_tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_prefix);
  if (workspace == nullptr || ws_bytes < need) return DTS_ERR_WORKSPACE;
  float *o_part = static_cast<float *>(workspace);
  float *lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + align_up(plan.o_bytes, 256));
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int page_shift = __builtin_ctz(static_cast<unsigned>(page_size));
  dts::RopeFreqs freqs;
  dts_host::make_rope_freqs(positions != nullptr ? rope_theta : 1.f, d, &freqs);

  if (max_prefix > 0) {
    CUtensorMap tk, tv;
    const int rpb = page_size < 128 ? page_size : 128;
    if (!make_cache_map(&tk, k_cache, d, Hkv, num_slots, rpb) || !make_cache_map(&tv, v_cache, d, Hkv, num_slots, rpb))
      return DTS_ERR_CUDA;
    PrefixArgs pa;
    pa.q = q;
    pa.page_table = page_table;
    pa.prefix_len = prefix_len;
    pa.positions = positions;
    pa.o_part = o_part;
    pa.lse_part = lse_part;
    pa.err = err_dev;
    pa.num_slots = num_slots;
    pa.max_prefix = max_prefix;
    pa.B = B;
    pa.N = N;
    pa.Hq = Hq;
    pa.Hkv = Hkv;
    pa.g = g;
    pa.M = N * g;
    pa.n_pairs = plan.n_pairs;
    pa.n_splits = plan.n_splits;
    pa.chunk = plan.chunk;
    pa.max_pages = max_pages;
    pa.page_shift = page_shift;
    pa.scale_log2 = scale * kLog2e;
    pa.freqs = freqs;
    const int64_t grid = static_cast<int64_t>(B) * Hkv * plan.n_splits * plan.n_pairs;
    if (grid >= (1ll << 31)) return DTS_ERR_UNSUPPORTED;
    const int st = d == 128 ? launch_prefix<128>(tk, tv, pa, static_cast<int>(grid), s)
                            : launch_prefix<64>(tk, tv, pa, static_cast<int>(grid), s);
    if (st != DTS_OK) return st;
  }

  WindowArgs wa;
  wa.q = q;
  wa.k_cache = k_cache;
  wa.v_cache = v_cache;
  wa.page_table = page_table;
  wa.prefix_len = prefix_len;
  wa.mask = mask;
  wa.positions = positions;
  wa.o_part = o_part;
  wa.lse_part = lse_part;
  wa.out = out;
  wa.lse2 = lse2;
  wa.err = err_dev;
  wa.num_slots = num_slots;
  wa.max_prefix = max_prefix;
  wa.B = B;
  wa.N = N;
  wa.Hq = Hq;
  wa.Hkv = Hkv;
  wa.g = g;
  wa.heads_per_warp = (g % 8 == 0) ? 8 : (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
  wa.max_pages = max_pages;
  wa.page_shift = page_shift;
  wa.n_splits = plan.n_splits;
  wa.chunk = plan.chunk;
  wa.scale_log2 = scale * kLog2e;
  wa.freqs = freqs;
  return d == 128 ? launch_window<128>(wa, s) : launch_window<64>(wa, s);
}
