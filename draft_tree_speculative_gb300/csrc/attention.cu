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
// Three kernels per call:
//
// 0. rope_q: rotates every query row once at its node's position and stores
//    it in bf16 (the model dtype) in the workspace.
//
// 1. prefix pass (tcgen05, persistent): the rows of a KV head are the N*g
//    (node, query head) pairs; a "unit" is (request, KV head, pair of 128-row
//    tiles), and its work is the ceil(P/128) key tiles of the request's prefix.
//    All units' key tiles form one flat sequence which the grid (one CTA per
//    SM) splits into equal contiguous ranges, so every SM gets the same work
//    whatever the prefix lengths. A CTA walks its range as segments (a unit's
//    tiles inside the range). Per segment, TMA brings the unit's Q tiles and
//    128-key K and V tiles (128-byte swizzle, one box per page and 64-column
//    block) into shared memory; one thread issues S = Q K^T into tensor memory;
//    each 128-thread softmax group owns one row tile (thread = TMEM lane =
//    row), turns S into bf16 P in place (P aliases the first half of S's
//    columns) and the MMA thread issues O += P V with P read from TMEM. The
//    running max is rescaled lazily (only when it grows by more than 2^8).
//    Each segment ends with a normalised fp32 partial O and its base-2 LSE
//    written to slot (unit + CTA index) of the workspace.
//
// 2. window + merge pass (SIMT): one warp per (node, KV head, head group).
//    It merges the unit's prefix segments by their LSEs (the CTAs that own the
//    unit's first and last tile bound them), then walks the set bits of the
//    node's ancestor mask (only those window keys are ever read, so
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
constexpr int kMaxGrid = 256;   // persistent CTAs: one per SM (GB300: 152), never more than this
int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int g, npt, rt, n_pairs, slot_rows;
  int64_t units, slots;
  int64_t o_off, lse_off, tb_off, q_off, total;
};

// Workspace: partial O [slots][slot_rows][d] fp32 | partial LSE
// [slots][slot_rows] fp32 | tiles-before table [B+1] int64 | rotated queries
// [B*N][Hq][d] bf16. A slot holds one unit's rows (at most two row tiles).
Plan make_plan(int B, int N, int Hq, int Hkv, int d) {
  Plan p;
  p.g = Hq / Hkv;
  p.npt = 128 / p.g;          // nodes per row tile
  p.rt = p.npt * p.g;         // rows per row tile (128 when g divides 128)
  const int M = N * p.g;
  p.n_pairs = (M + 2 * p.rt - 1) / (2 * p.rt);
  p.slot_rows = M < 2 * p.rt ? M : 2 * p.rt;
  p.units = static_cast<int64_t>(B) * Hkv * p.n_pairs;
  p.slots = p.units + kMaxGrid;
  p.o_off = 0;
  p.lse_off = align_up(p.o_off + p.slots * p.slot_rows * d * 4, 256);
  p.tb_off = align_up(p.lse_off + p.slots * p.slot_rows * 4, 256);
  p.q_off = align_up(p.tb_off + (static_cast<int64_t>(B) + 1) * 8, 256);
  p.total = align_up(p.q_off + static_cast<int64_t>(B) * N * Hq * d * 2, 256);
  return p;
}

// ============================================================================
// rope_q: q_rot[node][h] = bf16(RoPE(q[node][h], positions[node]))
// ============================================================================
struct RopeQArgs {
  const uint16_t *q;
  const int32_t *positions;
  uint16_t *q_rot;
  int rows, Hq, heads_per_thread;  // rows = B*N nodes
  dts::RopeFreqs freqs;
};

// One thread per (node, group of heads, 8-element chunk of the first half):
// the chunk's eight angles are computed once and applied to the group's heads.
// Consecutive threads take consecutive chunks of a row (coalesced 16-byte loads).
template <int D>
__global__ void __launch_bounds__(256) rope_q_kernel(const __grid_constant__ RopeQArgs a) {
  constexpr int kChunks = D / 16;
  const int hgroups = a.Hq / a.heads_per_thread;
  const int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (it >= static_cast<int64_t>(a.rows) * hgroups * kChunks) return;
  const int c = static_cast<int>(it % kChunks);
  const int hg = static_cast<int>((it / kChunks) % hgroups);
  const int64_t node = it / (static_cast<int64_t>(kChunks) * hgroups);
  const int pos = a.positions[node];
  float sn[8], cs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) dts::rope_sincos(pos, a.freqs.w[8 * c + e], &sn[e], &cs[e]);
  for (int hh = 0; hh < a.heads_per_thread; ++hh) {
    const int h = hg * a.heads_per_thread + hh;
    const int64_t off = (node * a.Hq + h) * D + 8 * c;
    uint4 x1 = *reinterpret_cast<const uint4 *>(a.q + off);
    uint4 x2 = *reinterpret_cast<const uint4 *>(a.q + off + D / 2);
    uint32_t *w1 = reinterpret_cast<uint32_t *>(&x1);
    uint32_t *w2 = reinterpret_cast<uint32_t *>(&x2);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float u0 = dts::bf16_lo(w1[e]), u1 = dts::bf16_hi(w1[e]);
      const float v0 = dts::bf16_lo(w2[e]), v1 = dts::bf16_hi(w2[e]);
      const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
      w1[e] = dts::pack_bf16x2(u0 * c0 - v0 * s0, u1 * c1 - v1 * s1);
      w2[e] = dts::pack_bf16x2(v0 * c0 + u0 * s0, v1 * c1 + u1 * s1);
    }
    *reinterpret_cast<uint4 *>(a.q_rot + off) = x1;
    *reinterpret_cast<uint4 *>(a.q_rot + off + D / 2) = x2;
  }
}

// ============================================================================
// prefix pass
// ============================================================================
struct PrefixArgs {
  const int32_t *page_table;
  const int32_t *prefix_len;
  float *o_part;
  float *lse_part;
  int64_t *tiles_before;  // [B + 1], written by CTA 0 for the merge pass
  int32_t *err;
  int64_t num_slots, max_prefix;
  int B, N, Hq, Hkv, g, M, rt, npt, n_pairs, slot_rows, max_pages, page_shift;
  float scale_log2;
};

template <int D>
struct PrefixShape {
  static constexpr int kThreads = 384;                 // 4 control warps + 2 softmax groups
  static constexpr uint32_t kTileBytes = 128 * D * 2;  // a 128-row bf16 tile (Q, K or V)
  static constexpr uint32_t kBlockBytes = 128 * 128;   // one 64-column block of a 128-row tile
  static constexpr int kSlots = D == 128 ? 5 : 8;      // K/V ring
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kSmem = 1024 /*align*/ + 2 * kTileBytes + kSlots * kTileBytes + kBarBytes;
};

// Key tiles of one unit of request b (0 for an empty or invalid prefix; the
// merge pass reports the invalid ones).
__device__ __forceinline__ int request_tiles(const int32_t *prefix_len, int b, int64_t max_prefix, int N,
                                             int max_pages, int page_shift) {
  const int P = prefix_len[b];
  if (P <= 0 || P > max_prefix || static_cast<int64_t>(P) + N > (static_cast<int64_t>(max_pages) << page_shift))
    return 0;
  return (P + 127) >> 7;
}

struct Segment {
  int b, hkv, pair, unit, lt0, lt1, P, nt;
};

// Walks the flat key-tile range [x, x1) as segments, in order.
struct SegmentWalker {
  int b;
  int nkt;
  int64_t tb;  // tiles of all units of requests < b
  int64_t x, x1;

  __device__ void init(const PrefixArgs &a, int64_t x0, int64_t x_end) {
    b = 0;
    tb = 0;
    nkt = a.B > 0 ? request_tiles(a.prefix_len, 0, a.max_prefix, a.N, a.max_pages, a.page_shift) : 0;
    x = x0;
    x1 = x_end;
  }
  __device__ bool next(const PrefixArgs &a, Segment &s) {
    if (x >= x1) return false;
    const int64_t per_req = static_cast<int64_t>(a.Hkv) * a.n_pairs;
    while (x >= tb + nkt * per_req) {
      tb += nkt * per_req;
      ++b;
      nkt = request_tiles(a.prefix_len, b, a.max_prefix, a.N, a.max_pages, a.page_shift);
    }
    const int64_t off = x - tb;
    const int uir = static_cast<int>(off / nkt);
    s.b = b;
    s.hkv = uir / a.n_pairs;
    s.pair = uir - s.hkv * a.n_pairs;
    s.unit = static_cast<int>(static_cast<int64_t>(b) * per_req + uir);
    s.lt0 = static_cast<int>(off - static_cast<int64_t>(uir) * nkt);
    s.lt1 = static_cast<int>(min(static_cast<int64_t>(nkt), s.lt0 + (x1 - x)));
    s.P = a.prefix_len[b];
    const int rows_left = a.M - s.pair * 2 * a.rt;
    s.nt = min(2, (rows_left + a.rt - 1) / a.rt);
    x += s.lt1 - s.lt0;
    return true;
  }
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    tree_prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ PrefixArgs a) {
  using S = PrefixShape<D>;
  constexpr int kSlots = S::kSlots;
  constexpr uint32_t kTileBytes = S::kTileBytes;
  constexpr int kKSteps = D / 16;  // K-steps of S = Q K^T
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

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
  uint64_t *o_free = o_fin + 2;
  uint64_t *q_full = o_free + 2;
  uint64_t *q_empty = q_full + 1;
  uint64_t *drain = q_empty + 1;
  int64_t *range = reinterpret_cast<int64_t *>(drain + 1);  // [0] = total tiles
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(range + 2);
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
      mbar_init(&o_free[t], 128);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // total key tiles over all units
    int64_t part = 0;
    for (int b = lane; b < a.B; b += 32)
      part += static_cast<int64_t>(request_tiles(a.prefix_len, b, a.max_prefix, a.N, a.max_pages, a.page_shift));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) range[0] = part * a.Hkv * a.n_pairs;
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_q);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (warp == 2 && blockIdx.x == 0 && lane == 0) {
    // tiles-before table for the merge pass
    int64_t acc = 0;
    for (int b = 0; b < a.B; ++b) {
      a.tiles_before[b] = acc;
      acc += static_cast<int64_t>(request_tiles(a.prefix_len, b, a.max_prefix, a.N, a.max_pages, a.page_shift)) *
             a.Hkv * a.n_pairs;
    }
    a.tiles_before[a.B] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t total = range[0];
  const int64_t x0 = total * blockIdx.x / gridDim.x;
  const int64_t x1 = total * (blockIdx.x + 1) / gridDim.x;
  const uint32_t sQ_addr = smem_addr(sQ);
  const uint32_t sKV_addr = smem_addr(sKV);
  SegmentWalker walker;
  walker.init(a, x0, x1);
  Segment sg;

  // Register split: the control warpgroup (TMA, MMA) gives registers to the
  // two softmax groups. 128 * 96 + 256 * 200 = 384 * 168, the launch budget.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;\n" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      // The whole warp walks the tiles; page ids come 32 at a time (one
      // coalesced load per 32 pages) and travel by shuffle; lane 0 issues.
      const int ps = 1 << a.page_shift;
      const int rows_per_box = ps < 128 ? ps : 128;
      const int boxes = 128 / rows_per_box;
      int use = 0, segc = 0;
      bool ok = true;
      while (ok && walker.next(a, sg)) {
        const int64_t pt_row = static_cast<int64_t>(sg.b) * a.max_pages;
        int batch_base = -(1 << 30);
        int my_pid = -1;
        // slot start of box r of the tile at kbase, or -1 (past the prefix or a bad page)
        auto box_slot = [&](int kbase, int nvalid, int r) -> int {
          if (r * rows_per_box >= nvalid) return -1;
          const int key = kbase + r * rows_per_box;
          const int pg = key >> a.page_shift;
          if (pg < batch_base || pg >= batch_base + 32) {  // warp-uniform
            batch_base = pg;
            my_pid = (pg + lane < a.max_pages) ? a.page_table[pt_row + pg + lane] : -1;
          }
          const int pid = __shfl_sync(0xffffffffu, my_pid, pg - batch_base);
          const int64_t s0 = static_cast<int64_t>(pid) * ps + (key & (ps - 1));
          if (pid < 0 || s0 + rows_per_box > a.num_slots) {
            if (lane == 0) dts::report(a.err, DTS_DEV_BAD_SLOT);
            return -1;
          }
          return static_cast<int>(s0);
        };
        // the unit's query tiles
        if (!mbar_wait(q_empty, (static_cast<uint32_t>(segc) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(q_full, static_cast<uint32_t>(sg.nt * (D / 64) * a.rt * 128));
          for (int t = 0; t < sg.nt; ++t) {
            const int node0 = (sg.pair * 2 + t) * a.npt;
            for (int h = 0; h < D / 64; ++h)
              tma_load_4d(sQ_addr + t * kTileBytes + h * S::kBlockBytes, &tm_q, h * 64, 0, sg.hkv,
                          sg.b * a.N + node0, q_full);
          }
        }
        ++segc;
        for (int lt = sg.lt0; lt < sg.lt1 && ok; ++lt) {
          const int kbase = lt * 128;
          const int nvalid = min(128, sg.P - kbase);
          int nbox = 0;
          for (int r = 0; r < boxes; ++r) nbox += box_slot(kbase, nvalid, r) >= 0 ? 1 : 0;
          for (int kv = 0; kv < 2; ++kv, ++use) {
            const int slot = use % kSlots;
            const uint32_t ph = static_cast<uint32_t>(use / kSlots) & 1u;
            if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (lane == 0)  // the barrier expects exactly the bytes of the boxes issued below
              mbar_expect_tx(&full[slot], static_cast<uint32_t>(nbox * rows_per_box * 128 * (D / 64)));
            const CUtensorMap *map = kv == 0 ? &tm_k : &tm_v;
            const uint32_t dst = sKV_addr + slot * kTileBytes;
            for (int r = 0; r < boxes; ++r) {
              const int s0 = box_slot(kbase, nvalid, r);
              if (s0 < 0 || lane != 0) continue;
              for (int h = 0; h < D / 64; ++h)
                tma_load_3d(dst + h * S::kBlockBytes + r * rows_per_box * 128, map, h * 64, sg.hkv, s0,
                            &full[slot]);
            }
            __syncwarp();
          }
        }
      }
      if (!ok) {
        if (lane == 0) {
          dts::report(a.err, DTS_DEV_TIMEOUT);
          // give the copies already in flight a bounded chance to land
          for (int u = max(0, use - kSlots); u < use; ++u)
            mbar_wait(&full[u % kSlots], static_cast<uint32_t>(u / kSlots) & 1u, abort_flag);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
      constexpr uint32_t kIdescO = idesc_bf16(128, D, true);
      auto slot_of = [](int use) { return use % kSlots; };
      auto phase_of = [](int use) { return static_cast<uint32_t>(use / kSlots) & 1u; };
      // One thread issues every MMA, so the issue loop must stay short: the
      // descriptors are built once and only their 16-byte start-address field
      // (bits 0-13) moves, by compile-time offsets, between MMAs.
      const uint64_t q_desc0 = sdesc_sw128(sQ_addr, 16, 1024);                // K-major Q tiles
      const uint64_t k_desc0 = sdesc_sw128(sKV_addr, 16, 1024);               // K-major K tiles
      const uint64_t v_desc0 = sdesc_sw128(sKV_addr, S::kBlockBytes, 1024);   // MN-major V tiles
      constexpr uint64_t kTileStep = kTileBytes >> 4;
      auto issue_s = [&](int t, int slot) {
        const uint64_t qa = q_desc0 + static_cast<uint64_t>(t) * kTileStep;
        const uint64_t kb = k_desc0 + static_cast<uint64_t>(slot) * kTileStep;
        const uint32_t d_tmem = tmem + t * 256;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
          const uint64_t off = ((ks >> 2) * S::kBlockBytes + (ks & 3) * 32) >> 4;
          mma_ss(d_tmem, qa + off, kb + off, kIdescS, ks > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int slot, bool first) {
        const uint64_t vb = v_desc0 + static_cast<uint64_t>(slot) * kTileStep;
        const uint32_t d_tmem = tmem + t * 256 + 128;
        const uint32_t p_tmem = tmem + t * 256;
        const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // 128 keys, 16 per step (2048 bytes of V)
          mma_ts(d_tmem, p_tmem + ks * 8, vb + static_cast<uint64_t>(ks) * (2048 >> 4), kIdescO, ks == 0 ? acc0 : 1u);
      };
      int use = 0, segc = 0;
      int tcnt[2] = {0, 0}, scnt[2] = {0, 0};
      bool ok = true;
      while (ok && walker.next(a, sg)) {
        const int nkt = sg.lt1 - sg.lt0;
        const int nt = sg.nt;
        // S for the segment's first tile needs its Q tiles and K
        ok = mbar_wait(q_full, static_cast<uint32_t>(segc) & 1u, abort_flag) &&
             mbar_wait(&full[slot_of(use)], phase_of(use), abort_flag);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          // (row-tile loops run over the constant 2 so that per-tile counters
          // stay in registers)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t < nt) {
              issue_s(t, slot_of(use));
              mma_commit(&s_full[t]);
            }
          }
          if (nkt == 1) mma_commit(q_empty);  // the segment's last S reads Q
          mma_commit(&empty[slot_of(use)]);
        }
        __syncwarp();
        // The tensor core takes about one group of MMAs at a time, so any work
        // between two issue calls leaves it idle. Per row tile all waits come
        // first; then PV_t(j) and S_t(j+1) go out back to back from one lane.
        for (int j = 0; j < nkt && ok; ++j) {
          const int vuse = use + 2 * j + 1;
          const int vslot = slot_of(vuse);
          const int kuse = use + 2 * (j + 1);
          const bool more = j + 1 < nkt;
          ok = mbar_wait(&full[vslot], phase_of(vuse), abort_flag) &&
               (!more || mbar_wait(&full[slot_of(kuse)], phase_of(kuse), abort_flag));
          if (!ok) break;
          const int nvalid = min(128, sg.P - (sg.lt0 + j) * 128);
          if (nvalid < 128) {
            // keys past the prefix's end: zero their V rows so that 0 * (stale or
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
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= nt) break;
            ok = mbar_wait(&p_full[t], static_cast<uint32_t>(tcnt[t] + j) & 1u, abort_flag);
            // the first PV of a segment overwrites O: the previous epilogue must have read it
            if (ok && j == 0 && scnt[t] > 0)
              ok = mbar_wait(&o_free[t], static_cast<uint32_t>(scnt[t] - 1) & 1u, abort_flag);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
              issue_pv(t, vslot, j == 0);
              if (more) issue_s(t, slot_of(kuse));  // overwrites P_t(j) only after PV_t(j) read it
              if (t == nt - 1) mma_commit(&empty[vslot]);
              if (more) {
                mma_commit(&s_full[t]);
                if (t == nt - 1) {
                  if (j + 2 == nkt) mma_commit(q_empty);
                  mma_commit(&empty[slot_of(kuse)]);
                }
              } else {
                mma_commit(&o_fin[t]);
              }
            }
            __syncwarp();
          }
        }
        use += 2 * nkt;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t < nt) {
            tcnt[t] += nkt;
            scnt[t] += 1;
          }
        }
        ++segc;
      }
      if (!ok) dts::report(a.err, DTS_DEV_TIMEOUT);
      // drain: wait for every MMA issued so far before TMEM is released
      if (lane == 0) mma_commit(drain);
      __syncwarp();
      mbar_wait(drain, 0, abort_flag);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;\n" ::: "memory");
    // ------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t tS = tmem + (static_cast<uint32_t>(wq * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    const float c = a.scale_log2;
    int tcnt = 0, scnt = 0;
    bool ok = true;
    while (ok && walker.next(a, sg)) {
      if (t >= sg.nt) continue;
      const int nkt = sg.lt1 - sg.lt0;
      const int prow = t * a.rt + r;                      // row within the unit's slot
      const int R = sg.pair * 2 * a.rt + prow;            // row of the KV head
      const bool warp_valid = wq * 32 < a.rt && sg.pair * 2 * a.rt + t * a.rt + wq * 32 < a.M;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkt; ++j) {
        if (!mbar_wait(&s_full[t], static_cast<uint32_t>(tcnt + j) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp_valid) {
          uint32_t sv[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sv[q]);
          tmem_wait_ld();
          const int nvalid = min(128, sg.P - (sg.lt0 + j) * 128);
          if (nvalid < 128) {  // the prefix's last tile: keys past its end score -inf
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (q * 32 + k >= nvalid) sv[q][k] = __float_as_uint(-INFINITY);
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              mx0 = max3(mx0, __uint_as_float(sv[q][k]), __uint_as_float(sv[q][k + 1]));
              mx1 = max3(mx1, __uint_as_float(sv[q][k + 2]), __uint_as_float(sv[q][k + 3]));
              mx2 = max3(mx2, __uint_as_float(sv[q][k + 4]), __uint_as_float(sv[q][k + 5]));
              mx3 = max3(mx3, __uint_as_float(sv[q][k + 6]), __uint_as_float(sv[q][k + 7]));
            }
          const float m_new = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
          float m_use = m_run;
          if (m_new > m_run + 8.f) m_use = m_new;  // lazy rescale: P stays below 2^8
          const float alpha = ex2(m_run - m_use);
          // P = 2^(s*c - m_use) as bf16 pairs, packed in place over the consumed
          // S registers: pair (q, k) lands in sv[q >> 1][(q & 1) * 16 + k / 2],
          // an entry already read. The scale-and-shift runs two lanes per FMA.
          const uint64_t cc = f2_pack(c, c);
          const uint64_t nm = f2_pack(-m_use, -m_use);
          uint64_t sum0 = f2_pack(0.f, 0.f), sum1 = sum0;
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
              const uint64_t x0 = ffma2(f2_pack(__uint_as_float(sv[q][k]), __uint_as_float(sv[q][k + 1])), cc, nm);
              const uint64_t x1v =
                  ffma2(f2_pack(__uint_as_float(sv[q][k + 2]), __uint_as_float(sv[q][k + 3])), cc, nm);
              float a0, a1, b0, b1;
              f2_unpack(x0, a0, a1);
              f2_unpack(x1v, b0, b1);
              a0 = ex2(a0);
              a1 = ex2(a1);
              b0 = ex2(b0);
              b1 = ex2(b1);
              sum0 = fadd2(sum0, f2_pack(a0, a1));
              sum1 = fadd2(sum1, f2_pack(b0, b1));
              sv[q >> 1][(q & 1) * 16 + (k >> 1)] = dts::pack_bf16x2(a0, a1);
              sv[q >> 1][(q & 1) * 16 + (k >> 1) + 1] = dts::pack_bf16x2(b0, b1);
            }
          float s00, s01, s10, s11;
          f2_unpack(sum0, s00, s01);
          f2_unpack(sum1, s10, s11);
          l_run = l_run * alpha + ((s00 + s01) + (s10 + s11));
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
      if (!ok || !mbar_wait(&o_fin[t], static_cast<uint32_t>(scnt) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (warp_valid) {
        const bool valid = r < a.rt && R < a.M;
        const int64_t slot_row = (static_cast<int64_t>(sg.unit) + blockIdx.x) * a.slot_rows + prow;
        const float inv_l = 1.f / l_run;
        float *dst = a.o_part + slot_row * D;
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
        if (valid) a.lse_part[slot_row] = m_run + __log2f(l_run);
      }
      tc_fence_before();
      mbar_arrive(&o_free[t]);
      tcnt += nkt;
      ++scnt;
    }
    if (!ok) dts::report(a.err, DTS_DEV_TIMEOUT);
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
  const uint16_t *q;  // rotated queries (bf16)
  const uint16_t *k_cache;
  const uint16_t *v_cache;
  const int32_t *page_table;
  const int32_t *prefix_len;
  const uint64_t *mask;
  const float *o_part;
  const float *lse_part;
  const int64_t *tiles_before;
  uint16_t *out;
  float *lse2;
  int32_t *err;
  int64_t num_slots, max_prefix;
  int B, N, Hq, Hkv, g, rt, n_pairs, slot_rows, heads_per_warp, max_pages, page_shift, grid, has_prefix;
  float scale_log2;
};

// Lane l holds elements {2l, 2l+1, D/2+2l, D/2+2l+1} (D = 128) or {l, D/2+l} (D = 64).
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
  const int i = static_cast<int>(node - static_cast<int64_t>(b) * a.N);
  const int h0 = hkv * a.g + hg * HW;
  const int P = a.prefix_len[b];

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

  float q[HW][E];
#pragma unroll
  for (int u = 0; u < HW; ++u) load_row<D>(a.q + (node * a.Hq + h0 + u) * D, lane, q[u]);

  float m[HW], l[HW], acc[HW][E];
#pragma unroll
  for (int u = 0; u < HW; ++u) {
    m[u] = -INFINITY;
    l[u] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[u][e] = 0.f;
  }

  // prefix segments of this row's unit: the CTAs that own the unit's first and
  // last key tile, and every one between, each left one partial in slot
  // (unit + CTA index). Largest LSE first, then an order-free weighted sum.
  const int nkt = a.has_prefix ? (P + 127) >> 7 : 0;
  if (nkt > 0) {
    const int64_t T = a.tiles_before[a.B];
    const int R = i * a.g + hg * HW;  // all HW heads share the pair
    const int pair = R / (2 * a.rt);
    const int prow0 = R - pair * 2 * a.rt;
    const int uir = hkv * a.n_pairs + pair;
    const int64_t unit = static_cast<int64_t>(b) * a.Hkv * a.n_pairs + uir;
    const int64_t start = a.tiles_before[b] + static_cast<int64_t>(uir) * nkt;
    const int64_t G = a.grid;
    const int64_t c_first = ((start + 1) * G - 1) / T;
    const int64_t c_last = ((start + nkt) * G - 1) / T;
    // with fewer tiles than CTAs some CTAs own no tile (and wrote no partial)
    auto owns_tiles = [&](int64_t cc) { return cc * T / G < (cc + 1) * T / G; };
    for (int64_t cc = c_first; cc <= c_last; ++cc) {
      if (!owns_tiles(cc)) continue;
      const int64_t base = (unit + cc) * a.slot_rows + prow0;
#pragma unroll
      for (int u = 0; u < HW; ++u) m[u] = fmaxf(m[u], a.lse_part[base + u]);
    }
#pragma unroll 2
    for (int64_t cc = c_first; cc <= c_last; ++cc) {
      if (!owns_tiles(cc)) continue;
      const int64_t base = (unit + cc) * a.slot_rows + prow0;
#pragma unroll
      for (int u = 0; u < HW; ++u) {
        const float wgt = dts::ptx::ex2(a.lse_part[base + u] - m[u]);
        const float *op = a.o_part + (base + u) * D;
        float x[E];
        if constexpr (D == 128) {
          const float2 lo2 = reinterpret_cast<const float2 *>(op)[lane];
          const float2 hi2 = reinterpret_cast<const float2 *>(op + 64)[lane];
          x[0] = lo2.x;
          x[1] = lo2.y;
          x[2] = hi2.x;
          x[3] = hi2.y;
        } else {
          x[0] = op[lane];
          x[1] = op[32 + lane];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[u][e] = fmaf(x[e], wgt, acc[u][e]);
        l[u] += wgt;
      }
    }
  }

  // window: the node's ancestors (and itself), in ascending node index
  const int ps = 1 << a.page_shift;
  uint64_t mk = a.mask[node];
  if (a.N < 64) mk &= (1ull << a.N) - 1;
  const int64_t pt_row = static_cast<int64_t>(b) * a.max_pages;
  // Ancestors go four at a time: their K/V rows are all in flight together,
  // and the four dot products of each head reduce across the warp side by side.
  constexpr int kBatch = 4;
  while (mk) {
    float kx[kBatch][E], vx[kBatch][E];
    bool have[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      have[k] = false;
      if (mk) {
        const int j = __ffsll(static_cast<long long>(mk)) - 1;
        mk &= mk - 1;
        const int64_t logical = static_cast<int64_t>(P) + j;
        const int pid = a.page_table[pt_row + (logical >> a.page_shift)];
        const int64_t slot = static_cast<int64_t>(pid) * ps + (logical & (ps - 1));
        if (pid < 0 || slot >= a.num_slots) {
          if (lane == 0) dts::report(a.err, DTS_DEV_BAD_SLOT);
        } else {
          load_row<D>(a.k_cache + (slot * a.Hkv + hkv) * D, lane, kx[k]);
          load_row<D>(a.v_cache + (slot * a.Hkv + hkv) * D, lane, vx[k]);
          have[k] = true;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < HW; ++u) {
      float s[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        float d = 0.f;
        if (have[k]) {
#pragma unroll
          for (int e = 0; e < E; ++e) d = fmaf(q[u][e], kx[k][e], d);
        }
        s[k] = d;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int k = 0; k < kBatch; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], o);
      float mn = m[u];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        s[k] *= a.scale_log2;
        if (have[k]) mn = fmaxf(mn, s[k]);
      }
      const float sa = mn == -INFINITY ? 1.f : dts::ptx::ex2(m[u] - mn);  // -inf: nothing seen yet
      l[u] *= sa;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[u][e] *= sa;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (!have[k]) continue;
        const float w = dts::ptx::ex2(s[k] - mn);
        l[u] += w;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[u][e] = fmaf(vx[k][e], w, acc[u][e]);
      }
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

bool encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (d, Hkv, slots) of a paged bf16 cache; box (64, 1, rows_per_box).
bool make_cache_map(CUtensorMap *map, const void *base, int d, int Hkv, int64_t num_slots, int rows_per_box) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_slots)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(rows_per_box)};
  return encode(map, base, 3, dims, strides, box);
}

// 4-D view (d, g, Hkv, B*N) of the queries [B*N][Hq][d]; box (64, g, 1, npt):
// one box holds the npt * g rows (node, head-in-group) of a row tile, in that order.
bool make_q_map(CUtensorMap *map, const void *base, int d, int g, int Hkv, int64_t nodes, int npt) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(nodes)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(g) * d * 2,
                           static_cast<cuuint64_t>(g) * Hkv * d * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(npt)};
  return encode(map, base, 4, dims, strides, box);
}

template <int D>
int launch_prefix(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const PrefixArgs &a, int grid,
                  cudaStream_t s) {
  using S = PrefixShape<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(tree_prefix_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(S::kSmem));
  });
  if (attr_err != cudaSuccess) return DTS_ERR_CUDA;
  tree_prefix_kernel<D><<<grid, S::kThreads, S::kSmem, s>>>(tk, tv, tq, a);
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
  if (B <= 0 || N < 1 || N > dts::kMaxNodes || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || Hq / Hkv > 128 ||
      (d != 64 && d != 128) || max_prefix < 0)
    return 0;
  return static_cast<size_t>(make_plan(B, N, Hq, Hkv, d).total);
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
  if (Hq / Hkv > 128) return DTS_ERR_UNSUPPORTED;
  if (page_size < 8 || page_size > 4096 || (page_size & (page_size - 1)) != 0) return DTS_ERR_UNSUPPORTED;
  if (max_prefix > (1ll << 30) || num_slots >= (1ll << 31)) return DTS_ERR_UNSUPPORTED;
  if (positions != nullptr && !(rope_theta > 0.f)) return DTS_ERR_INVALID;
  if (B == 0) return DTS_OK;
  if (!q || !k_cache || !v_cache || !page_table || !prefix_len || !mask || !out || !lse2) return DTS_ERR_INVALID;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
                       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out) |
                       reinterpret_cast<uintptr_t>(workspace);
  if (al & 15) return DTS_ERR_INVALID;
  if (static_cast<int64_t>(B) * N * Hq >= (1ll << 31) / d) return DTS_ERR_UNSUPPORTED;
  const Plan plan = make_plan(B, N, Hq, Hkv, d);
  if (workspace == nullptr || ws_bytes < static_cast<size_t>(plan.total)) return DTS_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  float *o_part = reinterpret_cast<float *>(ws + plan.o_off);
  float *lse_part = reinterpret_cast<float *>(ws + plan.lse_off);
  int64_t *tiles_before = reinterpret_cast<int64_t *>(ws + plan.tb_off);
  uint16_t *q_rot = reinterpret_cast<uint16_t *>(ws + plan.q_off);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int page_shift = __builtin_ctz(static_cast<unsigned>(page_size));
  const int g = Hq / Hkv;

  // 0. queries in the model dtype, rotated once
  const uint16_t *q_eff = q;
  if (positions != nullptr) {
    RopeQArgs ra;
    ra.q = q;
    ra.positions = positions;
    ra.q_rot = q_rot;
    ra.rows = B * N;
    ra.Hq = Hq;
    ra.heads_per_thread = (Hq % 4 == 0) ? 4 : (Hq % 2 == 0) ? 2 : 1;
    dts_host::make_rope_freqs(rope_theta, d, &ra.freqs);
    const int64_t items = static_cast<int64_t>(B) * N * (Hq / ra.heads_per_thread) * (d / 16);
    const int blocks = static_cast<int>((items + 255) / 256);
    if (d == 128) rope_q_kernel<128><<<blocks, 256, 0, s>>>(ra);
    else rope_q_kernel<64><<<blocks, 256, 0, s>>>(ra);
    if (dts_host::launch_status() != DTS_OK) return DTS_ERR_CUDA;
    q_eff = q_rot;
  }

  // 1. prefix pass, one CTA per SM
  int grid = 0;
  if (max_prefix > 0) {
    const int sms = dts_host::sm_count();
    grid = sms > 0 ? (sms < kMaxGrid ? sms : kMaxGrid) : 1;
    CUtensorMap tk, tv, tq;
    const int rpb = page_size < 128 ? page_size : 128;
    if (!make_cache_map(&tk, k_cache, d, Hkv, num_slots, rpb) || !make_cache_map(&tv, v_cache, d, Hkv, num_slots, rpb) ||
        !make_q_map(&tq, q_eff, d, g, Hkv, static_cast<int64_t>(B) * N, plan.npt))
      return DTS_ERR_CUDA;
    PrefixArgs pa;
    pa.page_table = page_table;
    pa.prefix_len = prefix_len;
    pa.o_part = o_part;
    pa.lse_part = lse_part;
    pa.tiles_before = tiles_before;
    pa.err = err_dev;
    pa.num_slots = num_slots;
    pa.max_prefix = max_prefix;
    pa.B = B;
    pa.N = N;
    pa.Hq = Hq;
    pa.Hkv = Hkv;
    pa.g = g;
    pa.M = N * g;
    pa.rt = plan.rt;
    pa.npt = plan.npt;
    pa.n_pairs = plan.n_pairs;
    pa.slot_rows = plan.slot_rows;
    pa.max_pages = max_pages;
    pa.page_shift = page_shift;
    pa.scale_log2 = scale * kLog2e;
    const int st = d == 128 ? launch_prefix<128>(tk, tv, tq, pa, grid, s) : launch_prefix<64>(tk, tv, tq, pa, grid, s);
    if (st != DTS_OK) return st;
  }

  // 2. window + merge pass
  WindowArgs wa;
  wa.q = q_eff;
  wa.k_cache = k_cache;
  wa.v_cache = v_cache;
  wa.page_table = page_table;
  wa.prefix_len = prefix_len;
  wa.mask = mask;
  wa.o_part = o_part;
  wa.lse_part = lse_part;
  wa.tiles_before = tiles_before;
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
  wa.rt = plan.rt;
  wa.n_pairs = plan.n_pairs;
  wa.slot_rows = plan.slot_rows;
  // at most 4 heads per warp: more warps in flight beat re-reading a few window rows
  wa.heads_per_warp = (g % 4 == 0) ? 4 : (g % 2 == 0) ? 2 : 1;
  wa.max_pages = max_pages;
  wa.page_shift = page_shift;
  wa.grid = grid;
  wa.has_prefix = grid > 0 ? 1 : 0;
  wa.scale_log2 = scale * kLog2e;
  return d == 128 ? launch_window<128>(wa, s) : launch_window<64>(wa, s);
}

// ============================================================================
// Allocation-free variant: the workspace is a fixed device array of this file.
//
// Some callers cannot hand out device memory: a process that has reserved the
// whole device for its own pool, a plugin with no access to its host's
// allocator, or code that must not call cudaMalloc while it runs. For them the
// workspace lives in this file-scope array instead. Every GPU that loads the
// library keeps the array for the life of the process.
// ============================================================================
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_ws_mutex;
void *g_static_ws_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device. The host-side
// name of the array is only a stand-in; its device address has to be asked
// for once per device, with that device current.
void *static_workspace(int *status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = DTS_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_static_ws_mutex);
  if (g_static_ws_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      *status = DTS_ERR_CUDA;
      return nullptr;
    }
    g_static_ws_ptr[dev] = p;
  }
  *status = DTS_OK;
  return g_static_ws_ptr[dev];
}

}  // namespace

extern "C" int dts_tree_verify_attention_static_ws(const uint16_t *q, const uint16_t *k_cache,
                                                   const uint16_t *v_cache, int64_t num_slots,
                                                   const int32_t *page_table, int max_pages, int page_size,
                                                   const int32_t *prefix_len, int64_t max_prefix,
                                                   const uint64_t *mask, const int32_t *positions, float rope_theta,
                                                   int B, int N, int Hq, int Hkv, int d, float softmax_scale,
                                                   uint16_t *out, float *lse2, int32_t *err_dev,
                                                   dts_stream_t stream) {
  if (B == 0) return DTS_OK;
  const size_t need = dts_tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_prefix);
  if (need > kStaticWorkspaceBytes) return DTS_ERR_WORKSPACE;
  int status = DTS_OK;
  void *ws = static_workspace(&status);
  if (ws == nullptr) return status;
  // No part of the workspace needs to start at zero: every byte a call reads
  // was written earlier in the same call.
  return dts_tree_verify_attention(q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                                   max_prefix, mask, positions, rope_theta, B, N, Hq, Hkv, d, softmax_scale, out,
                                   lse2, ws, kStaticWorkspaceBytes, err_dev, stream);
}
