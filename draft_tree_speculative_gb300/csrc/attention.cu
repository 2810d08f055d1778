// Tree-window attention: every query row attends the committed prefix plus
// the window keys its 64-bit mask selects. Verify: the N tree nodes are both
// the rows and the window (R = W = N), the mask holds the row's ancestors.
// Draft lanes: R = K lane rows over the (S - 1) * K-key lane window.
//
// [TS] "One tree attention": every row sees the committed prefix, and the
// 64-bit ancestor mask applies only to the window keys; the prefix is where
// the time goes at long context; results carry a base-2 log-sum-exp; draft
// lanes run the same with R = K over the lane window.
// [AK] section one: row v equals Target(prefix + path(root -> v)).
// [AK] section four: partial results over disjoint key sets merge by their
// log-sum-exps, O = sum Z_k O_k / sum Z_k.
//
// Three kernels per call:
//
// 0. prep: rotates every query row once at its node's position and stores it
//    in bf16 (the model dtype) in the workspace; writes NaN rows (and reports)
//    for requests whose prefix length is out of range.
//
// 1. tree attention (tcgen05, persistent): the rows of a KV head are the R*g
//    (row, query head) pairs; a "unit" is (request, KV head, pair of 128-row
//    tiles), and its keys are the P prefix keys followed by the W window keys
//    (the paged cache holds both), ceil((P + W)/128) key tiles. All units' key
//    tiles form one flat sequence which the grid (one CTA per SM) splits into
//    equal contiguous ranges, so every SM gets the same work whatever the
//    prefix lengths. A CTA walks its range as segments (a unit's tiles inside
//    the range). Per segment, TMA brings the unit's Q tiles and 128-key K and
//    V tiles (128-byte swizzle, one box per page and 64-column block) into
//    shared memory; one thread issues S = Q K^T into tensor memory; each
//    128-thread softmax group owns one row tile (thread = TMEM lane = row),
//    masks the window keys that are not the row's ancestors, turns S into
//    bf16 P in place (P aliases the first half of S's columns) and the MMA
//    thread issues O += P V with P read from TMEM. The running max is rescaled
//    lazily (only when it grows by more than 2^8).
//    A unit inside one segment writes its bf16 rows and base-2 LSEs directly.
//    Otherwise every segment writes a normalised fp32 partial O and its LSE
//    to slot (unit + CTA index).
//
// 2. merge (SIMT): for the units split over several CTAs, one warp per 8 rows
//    merges the partials by their LSEs (the CTAs that own the unit's first
//    and last tile bound them) and writes bf16 out and the fp32 base-2 LSE.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
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
  int64_t o_off, lse_off, tb_off, cnt_off, q_off, total;
};

// Workspace: partial O [slots][slot_rows][d] bf16 | partial LSE
// [slots][slot_rows] fp32 | tiles-before table [B+1] int64 | parts stored
// per unit [units] int32 | rotated queries [B*N][Hq][d] bf16. A slot holds
// one unit's rows (at most two row tiles).
Plan make_plan(int B, int R, int Hq, int Hkv, int d) {
  Plan p;
  p.g = Hq / Hkv;
  p.npt = 128 / p.g;          // nodes per row tile
  p.rt = p.npt * p.g;         // rows per row tile (128 when g divides 128)
  const int M = R * p.g;
  p.n_pairs = (M + 2 * p.rt - 1) / (2 * p.rt);
  p.slot_rows = M < 2 * p.rt ? M : 2 * p.rt;
  p.units = static_cast<int64_t>(B) * Hkv * p.n_pairs;
  p.slots = p.units + kMaxGrid;
  p.o_off = 0;
  p.lse_off = align_up(p.o_off + p.slots * p.slot_rows * d * 2, 256);
  p.tb_off = align_up(p.lse_off + p.slots * p.slot_rows * 4, 256);
  p.cnt_off = align_up(p.tb_off + (static_cast<int64_t>(B) + 1) * 8, 256);
  p.q_off = align_up(p.cnt_off + p.units * 4, 256);
  p.total = align_up(p.q_off + static_cast<int64_t>(B) * R * Hq * d * 2, 256);
  return p;
}

// ============================================================================
// prep: q_rot[node][h] = bf16(RoPE(q[node][h], positions[node])); NaN rows for
// out-of-range prefix lengths
// ============================================================================
struct PrepArgs {
  const uint16_t *q;
  const int32_t *positions;  // null: no rotation (q is used as given)
  const int32_t *prefix_len;
  uint16_t *q_rot;
  uint16_t *out;
  float *lse2;
  int32_t *err;
  int64_t max_prefix, capacity;  // capacity: page-table rows x page size
  int rows, R, W, Hq, heads_per_thread;   // rows = B*R query rows; W window keys per request
  int to_e4m3;  // FP8 cache: store the (rotated, bf16-rounded) queries as E4M3 bytes, and the
                // bf16 ones in `out` (read back there by the merge pass for the window keys)
  int32_t *unit_cnt;  // [units] zeroed here for the tree pass's merge (null: none)
  int64_t units;
  dts::RopeFreqs freqs;
};

// One thread per (node, group of heads, 8-element chunk of the first half):
// the chunk's eight angles are computed once and applied to the group's heads.
// Consecutive threads take consecutive chunks of a row (coalesced 16-byte loads).
template <int D>
__global__ void __launch_bounds__(256) attn_prep_kernel(const __grid_constant__ PrepArgs a) {
  dts::grid_dep_wait();
  dts::grid_dep_launch_next();
  constexpr int kChunks = D / 16;
  constexpr int kMaxHeads = 4;
  const int hgroups = a.Hq / a.heads_per_thread;
  const int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (a.unit_cnt != nullptr)
    for (int64_t u = it; u < a.units; u += static_cast<int64_t>(gridDim.x) * blockDim.x) a.unit_cnt[u] = 0;
  if (it >= static_cast<int64_t>(a.rows) * hgroups * kChunks) return;
  const int c = static_cast<int>(it % kChunks);
  const int hg = static_cast<int>((it / kChunks) % hgroups);
  const int64_t node = it / (static_cast<int64_t>(kChunks) * hgroups);
  const int64_t b = node / a.R;
  // every load up front: prefix length, position and the group's query chunks
  const int P = a.prefix_len[b];
  const int pos = a.positions != nullptr ? a.positions[node] : 0;
  uint4 x1[kMaxHeads], x2[kMaxHeads];
  if (a.positions != nullptr || a.to_e4m3) {
#pragma unroll
    for (int hh = 0; hh < kMaxHeads; ++hh) {
      if (hh >= a.heads_per_thread) break;
      const int64_t off = (node * a.Hq + hg * a.heads_per_thread + hh) * D + 8 * c;
      x1[hh] = *reinterpret_cast<const uint4 *>(a.q + off);
      x2[hh] = *reinterpret_cast<const uint4 *>(a.q + off + D / 2);
    }
  }
  if (P < 0 || P > a.max_prefix || static_cast<int64_t>(P) + a.W > a.capacity) {
    // the attention pass skips this request: its rows read NaN
    if (c == 0 && hg == 0 && node == b * a.R) dts::report(a.err, DTS_DEV_BAD_SLOT);
    const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    for (int hh = 0; hh < a.heads_per_thread; ++hh) {
      const int h = hg * a.heads_per_thread + hh;
      const int64_t off = (node * a.Hq + h) * D + 8 * c;
      *reinterpret_cast<uint4 *>(a.out + off) = nan4;
      *reinterpret_cast<uint4 *>(a.out + off + D / 2) = nan4;
      if (c == 0) a.lse2[node * a.Hq + h] = __int_as_float(0x7FC00000);
    }
    return;
  }
  if (a.positions == nullptr && !a.to_e4m3) return;
  float sn[8], cs[8];
  if (a.positions != nullptr) {
#pragma unroll
    for (int e = 0; e < 8; ++e) dts::rope_sincos(pos, a.freqs.w[8 * c + e], &sn[e], &cs[e]);
  }
#pragma unroll
  for (int hh = 0; hh < kMaxHeads; ++hh) {
    if (hh >= a.heads_per_thread) break;
    uint32_t *w1 = reinterpret_cast<uint32_t *>(&x1[hh]);
    uint32_t *w2 = reinterpret_cast<uint32_t *>(&x2[hh]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (a.positions != nullptr) {
        const float u0 = dts::bf16_lo(w1[e]), u1 = dts::bf16_hi(w1[e]);
        const float v0 = dts::bf16_lo(w2[e]), v1 = dts::bf16_hi(w2[e]);
        const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
        w1[e] = dts::pack_bf16x2(u0 * c0 - v0 * s0, u1 * c1 - v1 * s1);
        w2[e] = dts::pack_bf16x2(v0 * c0 + u0 * s0, v1 * c1 + u1 * s1);
      }
    }
    const int64_t off = (node * a.Hq + hg * a.heads_per_thread + hh) * D + 8 * c;
    if (a.to_e4m3) {
      // the bf16 values cast to E4M3 (nearest even, saturating): 8 bytes a half
      uint8_t *q8 = reinterpret_cast<uint8_t *>(a.q_rot);
      uint32_t b1[2], b2[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        b1[e] = dts::f32x2_to_e4m3x2(dts::bf16_lo(w1[2 * e]), dts::bf16_hi(w1[2 * e])) |
                (dts::f32x2_to_e4m3x2(dts::bf16_lo(w1[2 * e + 1]), dts::bf16_hi(w1[2 * e + 1])) << 16);
        b2[e] = dts::f32x2_to_e4m3x2(dts::bf16_lo(w2[2 * e]), dts::bf16_hi(w2[2 * e])) |
                (dts::f32x2_to_e4m3x2(dts::bf16_lo(w2[2 * e + 1]), dts::bf16_hi(w2[2 * e + 1])) << 16);
      }
      *reinterpret_cast<uint2 *>(q8 + off) = make_uint2(b1[0], b1[1]);
      *reinterpret_cast<uint2 *>(q8 + off + D / 2) = make_uint2(b2[0], b2[1]);
      *reinterpret_cast<uint4 *>(a.out + off) = x1[hh];
      *reinterpret_cast<uint4 *>(a.out + off + D / 2) = x2[hh];
      continue;
    }
    *reinterpret_cast<uint4 *>(a.q_rot + off) = x1[hh];
    *reinterpret_cast<uint4 *>(a.q_rot + off + D / 2) = x2[hh];
  }
}

// ============================================================================
// merge pass
// ============================================================================
struct MergeArgs {
  const uint16_t *o_part;  // bf16 partial rows
  const float *lse_part;
  const int64_t *tiles_before;
  const int32_t *prefix_len;
  uint16_t *out;
  float *lse2;
  int64_t max_prefix, capacity;
  int B, R, W, Hq, Hkv, g, M, rt, n_pairs, slot_rows, grid;  // W: window keys of the tree pass
  int owners32;  // every (tile index + 1) * groups fits in 32 bits
  // F8 only: the window part, from the bf16 rotated queries the prep pass
  // left in `out`, the mask and the E4M3 window K/V in the paged cache
  const uint64_t *mask;
  const uint8_t *k8, *v8;
  const int32_t *page_table;
  int32_t *err;
  int64_t num_slots;
  int Ww, max_pages, page_shift;  // Ww: window keys of the window part
  float scale_log2;
};

// Which group's range holds flat tile x, and whether group c owns any tile:
// the tree pass gives group c the tiles [c T / G, (c + 1) T / G).
struct Owners {
  int64_t T, G;
  bool w32;
  __device__ int64_t of(int64_t x) const {  // ((x + 1) G - 1) / T
    if (w32) return (static_cast<uint32_t>(x + 1) * static_cast<uint32_t>(G) - 1u) / static_cast<uint32_t>(T);
    return ((x + 1) * G - 1) / T;
  }
  __device__ bool owns(int64_t c) const {
    if (w32) {
      const uint32_t t = static_cast<uint32_t>(T), g = static_cast<uint32_t>(G), c32 = static_cast<uint32_t>(c);
      return c32 * t / g < (c32 + 1u) * t / g;
    }
    return c * T / G < (c + 1) * T / G;
  }
};

// The F8 merge of rows [64 blk, 64 blk + 64) of unit `unit` (row pair `pair`,
// request b, KV head hkv, prefix length P) by one CTA of eight warps, warp w
// taking 8 rows; lane 4 r + c of a warp holds its row r's columns
// {32 t + 8 c + u : t < 4, u < 8}. Each row first takes its visible window
// keys against its bf16 rotated query (left in `out` by the prep pass), with
// the E4M3 K and V rows widened exactly, in an online softmax in base 2
// (m, l, o). The window's K and V rows are copied into shared memory once
// for the CTA; a warp walks the union of its rows' visible keys, each row
// taking only the keys its mask holds. The prefix parts of the tree pass
// then join at the common maximum M: O = (2^(m - M) o + sum_k 2^(lse_k - M)
// O_k) / (2^(m - M) l + sum_k 2^(lse_k - M)), lse = M + log2 of that
// denominator. A non-finite K or V row turns the rows that see it NaN; a row
// whose window slot lies outside the cache reads NaN (after reporting).
__device__ __forceinline__ void merge_block_f8(const MergeArgs &a, uint32_t unit, int blk, int pair, int b, int hkv,
                                               int P, int64_t c_first, int64_t c_last, const Owners &own) {
  constexpr int D = 128;
  __shared__ __align__(128) uint8_t kv_s[2][dts::kMaxNodes * D];  // E4M3 window K | V rows
  __shared__ uint32_t bad_s[2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int prow = (blk * 8 + warp) * 8 + r;
  const int R = pair * 2 * a.rt + prow;  // row of the KV head
  const bool row_ok = prow < a.slot_rows;
  const bool valid = row_ok && R < a.M;
  const int node = valid ? R / a.g : 0;
  const int64_t node_row = static_cast<int64_t>(b) * a.R + node;
  const int64_t out_row = node_row * a.Hq + hkv * a.g + (R - node * a.g);
  const int64_t part_row = static_cast<int64_t>(unit) * a.slot_rows + prow;  // + part * slot_rows

  uint4 qv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    qv[t] = valid ? *reinterpret_cast<const uint4 *>(a.out + out_row * D + 32 * t + 8 * c) : make_uint4(0, 0, 0, 0);
  const uint64_t bits = valid ? a.mask[node_row] & (a.Ww < 64 ? (1ull << a.Ww) - 1ull : ~0ull) : 0ull;

  // pass 1: the largest LSE of the row's parts (lane c takes parts c, c + 4, ...;
  // the first four parts' LSEs are kept)
  float lse_first = -INFINITY, mx = -INFINITY;
  for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
    const int64_t part = c0 + c;
    float lse = -INFINITY;
    if (part <= c_last && row_ok && own.owns(part)) lse = a.lse_part[part_row + part * a.slot_rows];
    if (c0 == c_first) lse_first = lse;
    mx = fmaxf(mx, lse);
  }

  // the window's K and V rows into shared memory: warps 0 and 1 take keys
  // 32 w + lane, whose slots they look up and check
  if (warp < 2) {
    const int j = 32 * warp + lane;
    bool bad = false;
    if (j < a.Ww) {
      const int pos = P + j;
      const int page = a.page_table[static_cast<int64_t>(b) * a.max_pages + (pos >> a.page_shift)];
      const int64_t slot = (static_cast<int64_t>(page) << a.page_shift) + (pos & ((1 << a.page_shift) - 1));
      bad = page < 0 || slot >= a.num_slots;
      if (!bad) {
        const int64_t off = (slot * a.Hkv + hkv) * D;
#pragma unroll
        for (int x = 0; x < D / 16; ++x) {
          dts::ptx::cp_async_16(&kv_s[0][j * D + 16 * x], a.k8 + off + 16 * x);
          dts::ptx::cp_async_16(&kv_s[1][j * D + 16 * x], a.v8 + off + 16 * x);
        }
      }
    }
    const uint32_t bw = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) bad_s[warp] = bw;
    dts::ptx::cp_async_wait_all();
  }
  __syncthreads();
  if (!__any_sync(0xffffffffu, row_ok)) return;  // a warp past the slot's rows
  const uint64_t bad = a.Ww > 32 ? bad_s[0] | (static_cast<uint64_t>(bad_s[1]) << 32) : bad_s[0];

  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  uint64_t uni = bits;  // the window keys any of the warp's eight rows sees
  uni |= __shfl_xor_sync(0xffffffffu, uni, 4);
  uni |= __shfl_xor_sync(0xffffffffu, uni, 8);
  uni |= __shfl_xor_sync(0xffffffffu, uni, 16);
  if ((uni & bad) != 0ull && lane == 0) dts::report(a.err, DTS_DEV_BAD_SLOT);

  float m = -INFINITY, l = 0.f, o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;
  uint64_t todo = uni & ~bad;
  while (todo != 0ull) {
    const int j = __ffsll(static_cast<long long>(todo)) - 1;
    todo &= todo - 1ull;
    float dot = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint2 kw = *reinterpret_cast<const uint2 *>(&kv_s[0][j * D + 32 * t + 8 * c]);
      const uint32_t k01 = dts::e4m3x2_to_f16x2(kw.x & 0xFFFFu), k23 = dts::e4m3x2_to_f16x2(kw.x >> 16);
      const uint32_t k45 = dts::e4m3x2_to_f16x2(kw.y & 0xFFFFu), k67 = dts::e4m3x2_to_f16x2(kw.y >> 16);
      dot = fmaf(dts::bf16_lo(qv[t].x), dts::f16_lo(k01), dot);
      dot = fmaf(dts::bf16_hi(qv[t].x), dts::f16_hi(k01), dot);
      dot = fmaf(dts::bf16_lo(qv[t].y), dts::f16_lo(k23), dot);
      dot = fmaf(dts::bf16_hi(qv[t].y), dts::f16_hi(k23), dot);
      dot = fmaf(dts::bf16_lo(qv[t].z), dts::f16_lo(k45), dot);
      dot = fmaf(dts::bf16_hi(qv[t].z), dts::f16_hi(k45), dot);
      dot = fmaf(dts::bf16_lo(qv[t].w), dts::f16_lo(k67), dot);
      dot = fmaf(dts::bf16_hi(qv[t].w), dts::f16_hi(k67), dot);
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    if ((bits >> j) & 1ull) {
      const float sc = dot * a.scale_log2;
      const float m_new = fmaxf(m, sc);  // (a NaN score leaves m; its weight below is NaN)
      const float corr = m == -INFINITY ? 0.f : exp2f(m - m_new);
      const float p = sc == -INFINITY ? 0.f : exp2f(sc - m_new);
      l = l * corr + p;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint2 vw = *reinterpret_cast<const uint2 *>(&kv_s[1][j * D + 32 * t + 8 * c]);
        const uint32_t v01 = dts::e4m3x2_to_f16x2(vw.x & 0xFFFFu), v23 = dts::e4m3x2_to_f16x2(vw.x >> 16);
        const uint32_t v45 = dts::e4m3x2_to_f16x2(vw.y & 0xFFFFu), v67 = dts::e4m3x2_to_f16x2(vw.y >> 16);
        const float v[8] = {dts::f16_lo(v01), dts::f16_hi(v01), dts::f16_lo(v23), dts::f16_hi(v23),
                            dts::f16_lo(v45), dts::f16_hi(v45), dts::f16_lo(v67), dts::f16_hi(v67)};
#pragma unroll
        for (int u = 0; u < 8; ++u) o[8 * t + u] = o[8 * t + u] * corr + p * v[u];
      }
      m = m_new;
    }
  }

  // pass 2: the window sum and the parts at the common maximum
  const float M2 = fmaxf(mx, m);
  const float aw = m == -INFINITY ? 0.f : exp2f(m - M2);
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] *= aw;
  float den_parts = 0.f;  // this lane's parts (c, c + 4, ...)
  for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
    float lse = lse_first;
    if (c0 != c_first) {
      const int64_t part = c0 + c;
      lse = -INFINITY;
      if (part <= c_last && row_ok && own.owns(part)) lse = a.lse_part[part_row + part * a.slot_rows];
    }
    const float w = lse == -INFINITY ? 0.f : dts::ptx::ex2(lse - M2);  // a part that saw no key drops out
    den_parts += w;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (c0 + k > c_last) break;
      const float wk = __shfl_sync(0xffffffffu, w, (lane & ~3) | k);
      if (wk != 0.f) {
        const uint16_t *src = a.o_part + (part_row + (c0 + k) * a.slot_rows) * D + 8 * c;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint4 x = *reinterpret_cast<const uint4 *>(src + 32 * t);
          o[8 * t + 0] = fmaf(dts::bf16_lo(x.x), wk, o[8 * t + 0]);
          o[8 * t + 1] = fmaf(dts::bf16_hi(x.x), wk, o[8 * t + 1]);
          o[8 * t + 2] = fmaf(dts::bf16_lo(x.y), wk, o[8 * t + 2]);
          o[8 * t + 3] = fmaf(dts::bf16_hi(x.y), wk, o[8 * t + 3]);
          o[8 * t + 4] = fmaf(dts::bf16_lo(x.z), wk, o[8 * t + 4]);
          o[8 * t + 5] = fmaf(dts::bf16_hi(x.z), wk, o[8 * t + 5]);
          o[8 * t + 6] = fmaf(dts::bf16_lo(x.w), wk, o[8 * t + 6]);
          o[8 * t + 7] = fmaf(dts::bf16_hi(x.w), wk, o[8 * t + 7]);
        }
      }
    }
  }
  den_parts += __shfl_xor_sync(0xffffffffu, den_parts, 1);
  den_parts += __shfl_xor_sync(0xffffffffu, den_parts, 2);
  float den = aw * l + den_parts;  // (a NaN window sum stays NaN)
  if ((bits & bad) != 0ull) den = __int_as_float(0x7FC00000);
  if (!valid) return;
  const float inv = den == 0.f ? 0.f : 1.f / den;  // (a NaN sum stays NaN)
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint4 y;
    y.x = dts::pack_bf16x2(o[8 * t + 0] * inv, o[8 * t + 1] * inv);
    y.y = dts::pack_bf16x2(o[8 * t + 2] * inv, o[8 * t + 3] * inv);
    y.z = dts::pack_bf16x2(o[8 * t + 4] * inv, o[8 * t + 5] * inv);
    y.w = dts::pack_bf16x2(o[8 * t + 6] * inv, o[8 * t + 7] * inv);
    *reinterpret_cast<uint4 *>(a.out + out_row * D + 32 * t + 8 * c) = y;
  }
  if (c == 0) a.lse2[out_row] = den == 0.f ? -INFINITY : M2 + __log2f(den);
}

// The merge of rows [8 rb, 8 rb + 8) of unit `unit` (row pair `pair`, request
// b, KV head hkv, prefix length P) by one warp, from the parts left by the
// groups c_first .. c_last of the tree pass. kInPass: called by the tree pass
// itself, whose other CTAs stored the parts during the pass: their loads go to
// L2, past this SM's L1.
template <int D, bool kInPass = false>
__device__ __forceinline__ void merge_rows(const MergeArgs &a, uint32_t unit, int rb, int pair, int b, int hkv, int P,
                                           int64_t c_first, int64_t c_last, const Owners &own, int lane) {
  constexpr int kRows = 8;
  constexpr int E = D / 32;
  auto ld_part = [](const auto *p) {
    if constexpr (kInPass) return __ldcg(p);
    else return *p;
  };
  const int i_row = lane & 7;
  const int prow_l = rb * kRows + i_row;
  const bool row_ok = prow_l < a.slot_rows;
  const int64_t row0 = static_cast<int64_t>(unit) * a.slot_rows + prow_l;  // this lane's row in slot `unit`

  // pass 1: the largest LSE of each row (the first four parts' LSEs are kept)
  float lse_first = -INFINITY;
  float mx = -INFINITY;
  for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
    const int64_t c = c0 + (lane >> 3);
    float lse = -INFINITY;
    if (c <= c_last && row_ok && own.owns(c)) lse = ld_part(a.lse_part + row0 + c * a.slot_rows);
    if (c0 == c_first) lse_first = lse;
    mx = fmaxf(mx, lse);
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  // pass 2: weights, their sum and the weighted rows
  float acc[kRows][E];
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
  float den = 0.f;
  for (int64_t c0 = c_first; c0 <= c_last; c0 += 4) {
    const int64_t c = c0 + (lane >> 3);
    float lse = lse_first;
    if (c0 != c_first) {
      lse = -INFINITY;
      if (c <= c_last && row_ok && own.owns(c)) lse = ld_part(a.lse_part + row0 + c * a.slot_rows);
    }
    const float w = lse == -INFINITY ? 0.f : dts::ptx::ex2(lse - mx);  // a part that saw no key drops out
    den += w;
    // which of the four parts have rows to read (warp-uniform): a part whose
    // weights are all 0 (not a group with tiles, or no key seen) is skipped
    const uint32_t live = __ballot_sync(0xffffffffu, w != 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (((live >> (8 * k)) & 0xFFu) == 0u) continue;
      const uint16_t *base =
          a.o_part + ((static_cast<int64_t>(unit) + c0 + k) * a.slot_rows + rb * kRows) * D + E * lane;
      float x[kRows][E];
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (rb * kRows + i < a.slot_rows) {
          if constexpr (E == 4) {
            const uint2 v = ld_part(reinterpret_cast<const uint2 *>(base + i * D));
            x[i][0] = dts::bf16_lo(v.x);
            x[i][1] = dts::bf16_hi(v.x);
            x[i][2] = dts::bf16_lo(v.y);
            x[i][3] = dts::bf16_hi(v.y);
          } else {
            const uint32_t v = ld_part(reinterpret_cast<const unsigned int *>(base + i * D));
            x[i][0] = dts::bf16_lo(v);
            x[i][1] = dts::bf16_hi(v);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) x[i][e] = 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w, k * 8 + i);
        if (wi == 0.f) continue;  // warp-uniform
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = fmaf(x[i][e], wi, acc[i][e]);
      }
    }
  }
  den += __shfl_xor_sync(0xffffffffu, den, 8);
  den += __shfl_xor_sync(0xffffffffu, den, 16);

#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int prow = rb * kRows + i;
    const float den_i = __shfl_sync(0xffffffffu, den, i);
    const float mx_i = __shfl_sync(0xffffffffu, mx, i);
    const int R = pair * 2 * a.rt + prow;  // row of the KV head
    if (prow >= a.slot_rows || R >= a.M) continue;
    const int node = R / a.g;
    const int64_t node_row = static_cast<int64_t>(b) * a.R + node;
    const int64_t out_row = node_row * a.Hq + hkv * a.g + (R - node * a.g);
    const float inv = den_i == 0.f ? 0.f : 1.f / den_i;  // (a NaN sum stays NaN)
    if constexpr (E == 4) {
      uint2 v;
      v.x = dts::pack_bf16x2(acc[i][0] * inv, acc[i][1] * inv);
      v.y = dts::pack_bf16x2(acc[i][2] * inv, acc[i][3] * inv);
      *reinterpret_cast<uint2 *>(a.out + out_row * D + E * lane) = v;
    } else {
      *reinterpret_cast<uint32_t *>(a.out + out_row * D + E * lane) =
          dts::pack_bf16x2(acc[i][0] * inv, acc[i][1] * inv);
    }
    if (lane == 0) a.lse2[out_row] = den_i == 0.f ? -INFINITY : mx_i + __log2f(den_i);
  }
}


// ============================================================================
// tree attention
// ============================================================================
struct PrefixArgs {
  const int32_t *page_table;
  const int32_t *prefix_len;
  const uint64_t *mask;
  uint16_t *o_part;  // bf16 partial rows
  float *lse_part;
  int64_t *tiles_before;  // [B + 1], written by CTA 0 for the merge pass
  int32_t *unit_cnt;      // [units] parts of each unit stored so far (zeroed by prep); null: no merge here
  uint16_t *out;
  float *lse2;
  int32_t *err;
  int64_t num_slots, max_prefix;
  int B, R, W, Hq, Hkv, g, M, rt, npt, n_pairs, slot_rows, max_pages, page_shift;  // R rows, W window keys per request
  float scale_log2;
  long long wait_budget;  // cycles before a bounded wait gives up
  int stall;              // test hook: the producer issues no copy at all
  int owners32;           // every (tile index + 1) * grid fits in 32 bits
};

// A unit whose last part this CTA stored: the softmax groups merge it at the
// end of the pass.
struct MergeEntry {
  int64_t c_first, c_last;
  uint32_t unit;
  int pair, b, hkv, P, pad;
};

template <int D>
struct PrefixShape {
  static constexpr int kThreads = 384;                 // 4 control warps + 2 softmax groups
  static constexpr uint32_t kTileBytes = 128 * D * 2;  // a 128-row bf16 tile (Q, K or V)
  static constexpr uint32_t kBlockBytes = 128 * 128;   // one 64-column block of a 128-row tile
  static constexpr int kSlots = D == 128 ? 5 : 8;      // K/V ring
  static constexpr uint32_t kBarBytes = 512;
  // kfull, vfull, empty, vready rings, 10 single barriers, two poison masks,
  // then from the tile total on: 2 words for it, the TMEM address, the abort
  // flag and 3 counters (within 4 words), and 2 merge entries
  static_assert((4 * kSlots + 10) * 8 + 16 + 6 * 8 + 2 * sizeof(MergeEntry) <= kBarBytes, "barrier area too small");
  static constexpr uint32_t kSmem = 1024 /*align*/ + 2 * kTileBytes + kSlots * kTileBytes + kBarBytes;
};

// Key tiles of one unit of request b: prefix and window keys together (0 for
// a prefix length out of range; the prep kernel reports those).
__device__ __forceinline__ int request_tiles(const int32_t *prefix_len, int b, int64_t max_prefix, int W,
                                             int max_pages, int page_shift) {
  const int P = prefix_len[b];
  if (P < 0 || P > max_prefix || static_cast<int64_t>(P) + W > (static_cast<int64_t>(max_pages) << page_shift))
    return 0;
  return (P + W + 127) >> 7;
}

struct Segment {
  int b, hkv, pair, unit, lt0, lt1, P, nt, nkt;
  int64_t start;  // flat index of the unit's first key tile
};

// Walks the flat key-tile range [x, x1) as segments, in order. The flat
// order is (row pair, request, KV head, key tile): all units of the first
// 256 rows of every KV head, then those of the next 256 rows in the same
// order. With two pairs (M = 512) the two halves of the range mirror each
// other, so CTA c and CTA c + G/2 read the same K/V tiles at about the same
// time and the second read comes from L2.
struct SegmentWalker {
  int b;
  int nkt;
  int64_t tb;     // tiles of the units of requests < b within the current pair
  int64_t pbase;  // flat index of the current pair's first tile
  int64_t half;   // tiles of one pair (every request, every KV head)
  int64_t x, x1;

  __device__ void init(const PrefixArgs &a, int64_t x0, int64_t x_end, int64_t pair_tiles) {
    b = 0;
    tb = 0;
    half = pair_tiles;
    pbase = half > 0 ? x0 / half * half : 0;
    nkt = a.B > 0 ? request_tiles(a.prefix_len, 0, a.max_prefix, a.W, a.max_pages, a.page_shift) : 0;
    x = x0;
    x1 = x_end;
  }
  __device__ bool next(const PrefixArgs &a, Segment &s) {
    if (x >= x1) return false;
    while (x >= pbase + tb + static_cast<int64_t>(nkt) * a.Hkv) {
      tb += static_cast<int64_t>(nkt) * a.Hkv;
      if (++b == a.B) {  // the next pair's units
        b = 0;
        tb = 0;
        pbase += half;
      }
      nkt = request_tiles(a.prefix_len, b, a.max_prefix, a.W, a.max_pages, a.page_shift);
    }
    const int64_t off = x - pbase - tb;
    s.b = b;
    s.hkv = static_cast<int>(off / nkt);
    s.pair = static_cast<int>(pbase / half);
    // units numbered in the flat order, so that a partial's slot (unit + CTA
    // index) grows with the flat index and no two segments share one
    s.unit = (s.pair * a.B + b) * a.Hkv + s.hkv;
    s.nkt = nkt;
    s.start = pbase + tb + static_cast<int64_t>(s.hkv) * nkt;
    s.lt0 = static_cast<int>(off - static_cast<int64_t>(s.hkv) * nkt);
    s.lt1 = static_cast<int>(min(static_cast<int64_t>(nkt), s.lt0 + (x1 - x)));
    s.P = a.prefix_len[b];
    const int rows_left = a.M - s.pair * 2 * a.rt;
    s.nt = min(2, (rows_left + a.rt - 1) / a.rt);
    x += s.lt1 - s.lt0;
    return true;
  }
};

// Visibility of 32 consecutive keys to a row whose ancestor mask is mrow
// (bits >= N clear): bit k covers the key with window index o + k, i.e. a
// prefix key when o + k < 0 (always seen) and window key o + k otherwise
// (seen when that bit of mrow is set).
__device__ __forceinline__ uint32_t visible_word(int o, uint64_t mrow) {
  if (o <= -32) return ~0u;
  if (o >= 64) return 0u;
  if (o >= 0) return static_cast<uint32_t>(mrow >> o);
  return static_cast<uint32_t>(mrow << -o) | ((1u << -o) - 1u);
}

// P_t(r), the r-th key tile's P of row tile t (counted over the CTA's
// segments), passes from softmax group t to the MMA warp through a named
// barrier: the group's 128 threads arrive, the MMA warp syncs. Rounds r and
// r + 1 use different barriers, so a group that gives up can always arrive
// once more for the round the MMA warp may be waiting for (see the softmax
// groups) without landing in the round before it.
// Row tile 0's rounds also take warp 3, which vouches that V(j) is clean and
// K(j + 1) has landed before the MMA warp issues PV_0(j) and S_0(j + 1).
constexpr uint32_t kP0Threads = 128 + 32 + 32;
constexpr uint32_t kP1Threads = 128 + 32;
__device__ __forceinline__ uint32_t p_bar_threads(int t) { return t == 0 ? kP0Threads : kP1Threads; }
// Named-barrier operations are warp-aligned: the branches leading to them
// must be the same in every lane, so the result of a bounded wait that
// decides such a branch is taken for the whole warp.
__device__ __forceinline__ bool warp_all(bool x) { return __all_sync(0xffffffffu, x); }

__device__ __forceinline__ uint32_t p_bar_id(int t, int r) {
  return 1u + 2u * static_cast<uint32_t>(t) + (static_cast<uint32_t>(r) & 1u);
}
// The eight softmax warps meet once more, on their own barrier, before they
// merge the units whose last part the CTA stored.
constexpr uint32_t kMergeBarrier = 5;

// Phase of use u on a barrier that only the slot's uses of u's kind (K: even
// uses, V: odd ones) complete: with an even ring a slot holds the same kind
// every round, with an odd ring every other round.
template <int kSlots>
__device__ __forceinline__ uint32_t kind_phase(int use) {
  const int round = use / kSlots;
  return static_cast<uint32_t>(kSlots % 2 == 0 ? round : round >> 1) & 1u;
}

// Prepares the V tile of a tile that reaches the window (keys kbase ..
// kbase + 127, window index o = kbase - P of its first key) before any PV
// reads it, and returns the window keys whose V rows were not finite (as a
// mask over window indices, the same in every lane). Keys past the window's
// end get zero V rows, so that 0 * (stale or non-finite V) cannot reach O.
// Window keys are masked per row, so a row that does not see key x still
// multiplies P = 0 by x's V row: a non-finite V row there is zeroed and its
// key reported, and only the rows that see it turn NaN. Kept out of line so
// that the MMA warp's issue loop keeps its registers.
template <int D>
__device__ __forceinline__ uint64_t clean_window_v(uint8_t *vt, int o, int W, int lane) {
  constexpr uint32_t kBlockBytes = 128 * 128;
  const int nvalid = min(128, W - o);  // rows holding prefix or window keys
  for (int h = 0; h < D / 64; ++h) {
    uint4 *p = reinterpret_cast<uint4 *>(vt + h * kBlockBytes + nvalid * 128);
    const int n16 = (128 - nvalid) * 8;
    for (int e = lane; e < n16; e += 32) p[e] = make_uint4(0, 0, 0, 0);
  }
  uint64_t bad_keys = 0;
  for (int x = max(-o, 0) + lane; x < nvalid; x += 32) {
    bool bad = false;
    for (int h = 0; h < D / 64; ++h) {
      const uint4 *p = reinterpret_cast<const uint4 *>(vt + h * kBlockBytes + x * 128);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint4 v = p[e];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int f = 0; f < 4; ++f)
          bad |= ((w[f] & 0x7F80u) == 0x7F80u) || ((w[f] & 0x7F800000u) == 0x7F800000u);
      }
    }
    if (bad) {
      for (int h = 0; h < D / 64; ++h) {
        uint4 *p = reinterpret_cast<uint4 *>(vt + h * kBlockBytes + x * 128);
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = make_uint4(0, 0, 0, 0);
      }
      bad_keys |= 1ull << (o + x);
    }
  }
  fence_proxy_async();  // the zeroed rows are read by the tensor core
  __syncwarp();
  const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bad_keys));
  const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bad_keys >> 32));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// FP8 cache: widens, in place, rows [r0, r0 + 64) of the E4M3 V tile that
// TMA left in the slot's second half (128 rows of 128 bytes, 128-byte
// swizzle) into the layout of a bf16 tile (two 64-column blocks, same
// swizzle) holding f16 values, exact for every E4M3 value. Lane l takes rows
// r0 + l and r0 + l + 32 and reads a whole row before writing it; the row's
// second f16 block is the only place where its output overlaps the input,
// and that is the row's own bytes. Rows past the unit's keys become zero, and
// a window key (tile reaching the window, window index o of its first row)
// with a NaN byte gets a zero row and a bit in the returned mask, as
// clean_window_v does for a bf16 tile.
__device__ __forceinline__ uint64_t widen_fp8_v_rows(uint8_t *tile, int r0, int nvalid, int o, bool window,
                                                     int lane) {
  constexpr uint32_t kBlockBytes = 128 * 128;
  uint64_t bad_keys = 0;
#pragma unroll 1
  for (int x = r0 + lane; x < r0 + 64; x += 32) {
    const uint32_t sw = static_cast<uint32_t>(x & 7);
    uint4 *row0 = reinterpret_cast<uint4 *>(tile + x * 128);                // f16 columns 0..63
    uint4 *row1 = reinterpret_cast<uint4 *>(tile + kBlockBytes + x * 128);  // 64..127; the E4M3 row on entry
    if (x >= nvalid) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        row0[c] = make_uint4(0, 0, 0, 0);
        row1[c] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    uint4 in[8];  // 16-byte chunk c holds elements 16c .. 16c + 15
#pragma unroll
    for (int c = 0; c < 8; ++c) in[c] = row1[c ^ sw];
    bool zero = false;
    if (window && x >= -o) {
      uint32_t nan_bytes = 0;  // a byte whose low seven bits are all set (S.1111.111)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {in[c].x, in[c].y, in[c].z, in[c].w};
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const uint32_t t = (w[f] & 0x7F7F7F7Fu) ^ 0x7F7F7F7Fu;
          nan_bytes |= (t - 0x01010101u) & ~t & 0x80808080u;
        }
      }
      if (nan_bytes != 0u) {
        zero = true;
        bad_keys |= 1ull << (o + x);
      }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t w[4] = {in[c].x, in[c].y, in[c].z, in[c].w};
      uint32_t h[8];
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        h[2 * f] = zero ? 0u : dts::e4m3x2_to_f16x2(w[f] & 0xFFFFu);
        h[2 * f + 1] = zero ? 0u : dts::e4m3x2_to_f16x2(w[f] >> 16);
      }
      // elements 16c .. 16c + 15 are f16 chunks 2c and 2c + 1 of the row:
      // block c / 4, chunks 2 (c % 4) and 2 (c % 4) + 1 inside it
      uint4 *dst = c < 4 ? row0 : row1;
      const uint32_t c0 = 2u * static_cast<uint32_t>(c & 3);
      dst[c0 ^ sw] = make_uint4(h[0], h[1], h[2], h[3]);
      dst[(c0 + 1u) ^ sw] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  fence_proxy_async();  // the widened rows are read by the tensor core
  __syncwarp();
  const uint32_t lo = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bad_keys));
  const uint32_t hi = __reduce_or_sync(0xffffffffu, static_cast<uint32_t>(bad_keys >> 32));
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// F8: the K and V caches hold unscaled E4M3 bytes ([TS] "One tree attention",
// FP8 paragraph: no structural change; the prefix decode takes the query cast
// to FP8; the window kernel takes the unquantized query and widens the
// window's FP8 K/V after loading). This pass then covers the prefix keys only
// (the host passes W = 0) and leaves a partial for every unit; the merge pass
// adds the window keys. S = Q K^T runs as an FP8 MMA (kind::f8f6f4) on the
// E4M3 query (rotated, rounded to bf16, then cast) and the K tile as loaded.
// Warps 2 and 3 widen each V tile to f16 in shared memory (64 rows each), and
// O += P V runs in f16 with P in f16.
template <int D, bool F8>
__global__ void __launch_bounds__(384, 1)
    tree_prefix_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ PrefixArgs a) {
  dts::grid_dep_wait();
  dts::grid_dep_launch_next();
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
  // The ring's slots hold K and V tiles in turn (use u: K when even, V when
  // odd). A load completes on kfull or vfull by its kind, so each of those
  // barriers is waited by one role only, at consecutive phases.
  uint64_t *kfull = bars;
  uint64_t *vfull = bars + kSlots;
  uint64_t *empty = bars + 2 * kSlots;
  uint64_t *s_full = bars + 3 * kSlots;
  uint64_t *o_fin = s_full + 2;
  uint64_t *o_free = o_fin + 2;
  uint64_t *q_full = o_free + 2;
  uint64_t *q_empty = q_full + 1;
  uint64_t *drain = q_empty + 1;
  uint64_t *win_bar = drain + 1;                             // the segment's poisoned-key mask is written
  uint64_t *vready = win_bar + 1;                            // [kSlots] a V tile landed and is clean
  uint64_t *poison = vready + kSlots;                        // [2] window keys whose V rows were not finite
  int64_t *range = reinterpret_cast<int64_t *>(poison + 2);  // [0] = total tiles
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(range + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // [0], [1]: warps of the CTA's first / last partial segment that stored
  // their rows; [2]: entries in the merge list
  int *part_cnt = const_cast<int *>(abort_flag) + 1;
  MergeEntry *mlist = reinterpret_cast<MergeEntry *>(range + 6);  // [2]

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&o_fin[t], 1);
      mbar_init(&o_free[t], 128);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(drain, 1);
    // F8: both V warps (2 and 3) arrive on vready and win_bar
    mbar_init(win_bar, F8 ? 2 : 1);
    for (int s2 = 0; s2 < kSlots; ++s2) mbar_init(&vready[s2], F8 ? 2 : 1);
    poison[1] = 0;
    *abort_flag = 0;
    part_cnt[0] = part_cnt[1] = part_cnt[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    // total key tiles over all units
    int64_t part = 0;
    for (int b = lane; b < a.B; b += 32)
      part += static_cast<int64_t>(request_tiles(a.prefix_len, b, a.max_prefix, a.W, a.max_pages, a.page_shift));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) range[0] = part * a.Hkv * a.n_pairs;  // n_pairs mirror-image halves
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
  if (warp == 3 && blockIdx.x == 0 && lane == 0) {
    // tiles-before table for the merge pass (within one row pair; the last
    // entry is the tiles of one pair)
    int64_t acc = 0;
    for (int b = 0; b < a.B; ++b) {
      a.tiles_before[b] = acc;
      acc += static_cast<int64_t>(request_tiles(a.prefix_len, b, a.max_prefix, a.W, a.max_pages, a.page_shift)) *
             a.Hkv;
    }
    a.tiles_before[a.B] = acc;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long wait_budget = a.wait_budget;
  const int64_t total = range[0];
  const int64_t x0 = total * blockIdx.x / gridDim.x;
  const int64_t x1 = total * (blockIdx.x + 1) / gridDim.x;
  const uint32_t sQ_addr = smem_addr(sQ);
  const uint32_t sKV_addr = smem_addr(sKV);
  SegmentWalker walker;
  walker.init(a, x0, x1, total / a.n_pairs);
  Segment sg;

  // Register split: the control warpgroup (TMA, MMA) gives registers to the
  // two softmax groups: 128 * 112 + 256 * 192 = 63 488 <= 384 * 168, the
  // launch budget. Below 112 the control roles' loops spill to local memory,
  // which every barrier wait of the MMA warp then pays for.
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 112;\n" ::: "memory");
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      // The whole warp walks the tiles; page ids come 32 at a time (one
      // coalesced load per 32 pages) and travel by shuffle; lane 0 issues.
      const int ps = 1 << a.page_shift;
      const int rows_per_box = ps < 128 ? ps : 128;
      const int boxes = 128 / rows_per_box;
      // a Q, K or V row is D / 64 boxes of 64 bf16 columns, or one box of
      // D = 128 E4M3 bytes; an E4M3 V tile lands in the slot's second half, to
      // be widened there
      constexpr int kRowBoxes = F8 ? 1 : D / 64;
      int use = 0, segc = 0;
      bool ok = true;
      // (a.stall, a test hook: no copy is ever issued, so the consumers' waits
      // run out and the kernel leaves with DTS_DEV_TIMEOUT)
      while (ok && a.stall == 0 && walker.next(a, sg)) {
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
        if (!mbar_wait(q_empty, (static_cast<uint32_t>(segc) & 1u) ^ 1u, abort_flag, wait_budget)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_expect_tx(q_full, static_cast<uint32_t>(sg.nt * kRowBoxes * a.rt * 128));
          for (int t = 0; t < sg.nt; ++t) {
            const int node0 = (sg.pair * 2 + t) * a.npt;
            for (int h = 0; h < kRowBoxes; ++h)
              tma_load_4d(sQ_addr + t * kTileBytes + h * S::kBlockBytes, &tm_q, h * 64, 0, sg.hkv,
                          sg.b * a.R + node0, q_full);
          }
        }
        ++segc;
        for (int lt = sg.lt0; lt < sg.lt1 && ok; ++lt) {
          const int kbase = lt * 128;
          const int nvalid = min(128, sg.P + a.W - kbase);
          int nbox = 0;
          for (int r = 0; r < boxes; ++r) nbox += box_slot(kbase, nvalid, r) >= 0 ? 1 : 0;
          for (int kv = 0; kv < 2; ++kv, ++use) {
            const int slot = use % kSlots;
            const uint32_t ph = static_cast<uint32_t>(use / kSlots) & 1u;
            if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag, wait_budget)) {
              ok = false;
              break;
            }
            uint64_t *done = kv == 0 ? &kfull[slot] : &vfull[slot];
            if (lane == 0)  // the barrier expects exactly the bytes of the boxes issued below
              mbar_expect_tx(done, static_cast<uint32_t>(nbox * rows_per_box * 128 * kRowBoxes));
            const CUtensorMap *map = kv == 0 ? &tm_k : &tm_v;
            const uint32_t dst = sKV_addr + slot * kTileBytes + (F8 && kv == 1 ? S::kBlockBytes : 0u);
            for (int r = 0; r < boxes; ++r) {
              const int s0 = box_slot(kbase, nvalid, r);
              if (s0 < 0 || lane != 0) continue;
              for (int h = 0; h < kRowBoxes; ++h)
                tma_load_3d(dst + h * S::kBlockBytes + r * rows_per_box * 128, map, h * 64, sg.hkv, s0, done);
            }
            __syncwarp();
          }
        }
      }
      if (!ok) {
        if (lane == 0) {
          dts::report(a.err, DTS_DEV_TIMEOUT);
          // the copies already in flight land before the CTA's shared memory
          // goes (bounded, whatever the abort flag says)
          for (int u = max(0, use - kSlots); u < use; ++u)
            mbar_wait_own((u & 1) ? &vfull[u % kSlots] : &kfull[u % kSlots], kind_phase<kSlots>(u), wait_budget);
          if (segc > 0) mbar_wait_own(q_full, static_cast<uint32_t>(segc - 1) & 1u, wait_budget);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescS = F8 ? idesc_f16(128, 128, false) : idesc_bf16(128, 128, false);  // F8: E4M3
      constexpr uint32_t kIdescO = F8 ? idesc_f16(128, D, true) : idesc_bf16(128, D, true);
      auto slot_of = [](int use) { return use % kSlots; };
      auto kind_phase_of = [](int use) { return kind_phase<kSlots>(use); };
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
        if constexpr (F8) {
          // one 128-byte E4M3 row per query and key: four K-steps of 32
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_ss_f8(d_tmem, qa + ks * 2, kb + ks * 2, kIdescS, ks > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int ks = 0; ks < kKSteps; ++ks) {
            const uint64_t off = ((ks >> 2) * S::kBlockBytes + (ks & 3) * 32) >> 4;
            mma_ss(d_tmem, qa + off, kb + off, kIdescS, ks > 0 ? 1u : 0u);
          }
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
      int tcnt[2] = {0, 0};
      int p0_rounds = 0;  // rounds of row tile 0 this warp has synced
      bool ok = true;
      while (ok && walker.next(a, sg)) {
        const int nkt = sg.lt1 - sg.lt0;
        const int nt = sg.nt;
        // S for the segment's first tile needs its Q tiles and K
        ok = warp_all(mbar_wait(q_full, static_cast<uint32_t>(segc) & 1u, abort_flag, wait_budget) &&
                      mbar_wait(&kfull[slot_of(use)], kind_phase_of(use), abort_flag, wait_budget));
        if (!ok) break;
        tc_fence_after();
        int kslot = slot_of(use);  // the slot of K(j + 1) in the loop below, of K(0) here
        if (lane == 0) {
          // (row-tile loops run over the constant 2 so that per-tile counters
          // stay in registers)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t < nt) {
              issue_s(t, kslot);
              mma_commit(&s_full[t]);
            }
          }
          if (nkt == 1) mma_commit(q_empty);  // the segment's last S reads Q
          mma_commit(&empty[kslot]);
        }
        __syncwarp();
        int vslot = kslot + 1 == kSlots ? 0 : kslot + 1;  // V(j)
        // The tensor core takes about one MMA at a time from the issuing
        // thread, so whatever that thread does between two groups leaves it
        // idle; an mbarrier wait costs it ~135 cycles even on a completed
        // phase, a named-barrier sync ~15. So the one wait per row tile and
        // key tile is a named-barrier sync, after which PV_t(j) and S_t(j+1)
        // go out back to back from one lane, and the abort flag read before
        // them is looked at only after them.
        for (int j = 0; j < nkt && ok; ++j) {
          kslot = vslot + 1 == kSlots ? 0 : vslot + 1;  // K(j + 1)
          const bool more = j + 1 < nkt;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= nt) break;
            // Group t has stored P_t(j) in TMEM and, on a segment's first
            // tile, read O_t of the previous segment (which PV_t(0)
            // overwrites). In row tile 0's rounds warp 3 vouches for V(j)
            // and K(j + 1). A warp that gives up sets the abort flag before
            // its last arrival.
            named_sync(p_bar_id(t, tcnt[t] + j), p_bar_threads(t));
            if (t == 0) ++p0_rounds;
            const int aborted = *abort_flag;
            tc_fence_after();
            if (lane == 0) {
              issue_pv(t, vslot, j == 0);
              if (more) issue_s(t, kslot);  // overwrites P_t(j) only after PV_t(j) read it
              if (t == nt - 1) mma_commit(&empty[vslot]);
              if (more) {
                mma_commit(&s_full[t]);
                if (t == nt - 1) {
                  if (j + 2 == nkt) mma_commit(q_empty);
                  mma_commit(&empty[kslot]);
                }
              } else {
                mma_commit(&o_fin[t]);
              }
            }
            __syncwarp();
            if (aborted) {
              ok = false;
              break;
            }
          }
          vslot = kslot + 1 == kSlots ? 0 : kslot + 1;  // V(j + 1)
        }
        use += 2 * nkt;
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (t < nt) tcnt[t] += nkt;
        ++segc;
      }
      if (!ok) {
        // warp 3 may be blocked in row tile 0's round p0_rounds, which this
        // warp has not joined; the abort flag is set, so one more arrival
        // ends that sync and warp 3 stops there
        named_arrive(p_bar_id(0, p0_rounds), kP0Threads);
        dts::report(a.err, DTS_DEV_TIMEOUT);
      }
      // drain: wait for every MMA issued so far before TMEM is released
      if (lane == 0) mma_commit(drain);
      __syncwarp();
      mbar_wait_own(drain, 0, wait_budget);
    } else {
      // ---------------------------------------------------------- V-tile warp(s), voucher
      // Warp 2 (and warp 3 under F8) hands every V tile on (vready) once it
      // has landed, after cleaning the ones that reach the window
      // (clean_window_v), and publishes each segment's poisoned window keys
      // (win_bar). F8: warps 2 and 3 each widen half of every V tile's rows
      // and publish their own mask. Warp 3 also vouches, in row tile 0's
      // round j, that V(j) is ready and K(j + 1) has landed, so that the MMA
      // warp waits only on the named barrier.
      const bool v_role = warp == 2 || F8;
      const bool voucher = warp == 3;
      const int vw = warp - 2;
      int use = 0, prev_nt = 0;
      int rounds = 0;        // row tile 0 rounds this warp has synced (voucher)
      int scnt[2] = {0, 0};  // segments each softmax group has taken part in
      bool ok = true;
      while (ok && walker.next(a, sg)) {
        const int nkt = sg.lt1 - sg.lt0;
        uint64_t seg_poison = 0;
        for (int j = 0; j < nkt && ok; ++j) {
          const int vuse = use + 2 * j + 1;
          const int vslot = vuse % kSlots;
          if (v_role) {
            ok = warp_all(mbar_wait(&vfull[vslot], kind_phase<kSlots>(vuse), abort_flag, wait_budget));
            if (!ok) break;
            const int kbase = (sg.lt0 + j) * 128;
            if constexpr (F8) {
              seg_poison |= widen_fp8_v_rows(sKV + vslot * kTileBytes, vw * 64, min(128, sg.P + a.W - kbase),
                                             kbase - sg.P, kbase + 128 > sg.P, lane);
            } else if (kbase + 128 > sg.P) {  // the window's tiles (and the unit's end)
              seg_poison |= clean_window_v<D>(sKV + vslot * kTileBytes, kbase - sg.P, a.W, lane);
            }
            if (lane == 0) mbar_arrive(&vready[vslot]);
            __syncwarp();
          }
          if (voucher) {
            const int kuse = vuse + 1;
            ok = warp_all(mbar_wait(&vready[vslot], kind_phase<kSlots>(vuse), abort_flag, wait_budget) &&
                          (j + 1 == nkt ||
                           mbar_wait(&kfull[kuse % kSlots], kind_phase<kSlots>(kuse), abort_flag, wait_budget)));
            if (!ok) break;
            named_sync(p_bar_id(0, rounds), kP0Threads);
            ++rounds;
            if (*abort_flag) {
              ok = false;
              break;
            }
          }
        }
        if (v_role) {
          // The groups that read the previous segment's mask must be past it
          // (o_free follows their read) before it is overwritten.
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (ok && t < prev_nt && scnt[t] > 0)
              ok = warp_all(mbar_wait(&o_free[t], static_cast<uint32_t>(scnt[t] - 1) & 1u, abort_flag, wait_budget));
          prev_nt = sg.nt;
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (t < sg.nt) ++scnt[t];
          if (lane == 0) {
            poison[vw] = seg_poison;
            mbar_arrive(win_bar);
          }
          __syncwarp();
        }
        use += 2 * nkt;
      }
      if (!ok) {
        // the MMA warp may be blocked in row tile 0's round `rounds`: one
        // more arrival (the abort flag is set) ends it there
        if (voucher) named_arrive(p_bar_id(0, rounds), kP0Threads);
        dts::report(a.err, DTS_DEV_TIMEOUT);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory");
    // ------------------------------------------------------------ softmax groups
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t tS = tmem + (static_cast<uint32_t>(wq * 32) << 16) + t * 256;
    const uint32_t tO = tS + 128;
    const float c = a.scale_log2;
    const uint64_t node_bits = a.W < 64 ? (1ull << a.W) - 1ull : ~0ull;  // the window's keys
    int tcnt = 0, scnt = 0, wcnt = 0;
    int arrived = 0;  // this warp's arrivals on the P barriers: the next round is `arrived`
    bool ok = true;
    while (ok && walker.next(a, sg)) {
      const uint32_t wpar = static_cast<uint32_t>(wcnt++) & 1u;  // win_bar completes once per segment
      // the unit lies inside this segment (F8: the merge pass adds the window
      // keys to every unit, so every unit leaves a partial)
      const bool whole = !F8 && sg.lt0 == 0 && sg.lt1 == sg.nkt;
      if (t >= sg.nt) continue;
      const int nkt = sg.lt1 - sg.lt0;
      const int prow = t * a.rt + r;                      // row within the unit's slot
      const int R = sg.pair * 2 * a.rt + prow;            // row of the KV head
      const bool warp_valid = wq * 32 < a.rt && sg.pair * 2 * a.rt + t * a.rt + wq * 32 < a.M;
      const bool valid = warp_valid && r < a.rt && R < a.M;
      // the row's ancestor mask (bits >= N clear), read where a tile reaches the window
      auto row_mask = [&]() -> uint64_t {
        return valid ? (a.mask[static_cast<int64_t>(sg.b) * a.R + R / a.g] & node_bits) : 0ull;
      };
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkt; ++j) {
        const bool in_window = (sg.lt0 + j) * 128 + 128 > sg.P;
        uint64_t mrow = 0;
        if (in_window) mrow = row_mask();  // in flight during the wait below
        if (!warp_all(mbar_wait(&s_full[t], static_cast<uint32_t>(tcnt + j) & 1u, abort_flag, wait_budget))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp_valid) {
          uint32_t sv[4][32];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sv[q]);
          tmem_wait_ld();
          const int kbase = (sg.lt0 + j) * 128;
          if (in_window) {
            // the window's tiles: a key counts only if the row may see it
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t vis = visible_word(kbase + q * 32 - sg.P, mrow);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                if (!(vis & (1u << k))) sv[q][k] = __float_as_uint(-INFINITY);
            }
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
          // a row may see no key of a tile (or of a whole segment): m_use stays
          // -inf, P is 0 and nothing rescales
          const float m_sub = m_use == -INFINITY ? 0.f : m_use;
          const float alpha = m_use == -INFINITY ? 1.f : ex2(m_run - m_use);
          // P = 2^(s*c - m_use) as bf16 pairs (f16 under F8), packed in place over the consumed
          // S registers: pair (q, k) lands in sv[q >> 1][(q & 1) * 16 + k / 2],
          // an entry already read. The scale-and-shift runs two lanes per FMA.
          const uint64_t cc = f2_pack(c, c);
          const uint64_t nm = f2_pack(-m_sub, -m_sub);
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
              if constexpr (F8) {
                sv[q >> 1][(q & 1) * 16 + (k >> 1)] = dts::pack_f16x2(a0, a1);
                sv[q >> 1][(q & 1) * 16 + (k >> 1) + 1] = dts::pack_f16x2(b0, b1);
              } else {
                sv[q >> 1][(q & 1) * 16 + (k >> 1)] = dts::pack_bf16x2(a0, a1);
                sv[q >> 1][(q & 1) * 16 + (k >> 1) + 1] = dts::pack_bf16x2(b0, b1);
              }
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
        named_arrive(p_bar_id(t, arrived), p_bar_threads(t));
        ++arrived;
      }
      if (!ok || !warp_all(mbar_wait(&o_fin[t], static_cast<uint32_t>(scnt) & 1u, abort_flag, wait_budget) &&
                           mbar_wait(win_bar, wpar, abort_flag, wait_budget))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // a row that sees a window key whose V row was not finite reads NaN
      const uint64_t seg_poison = F8 ? (poison[0] | poison[1]) : poison[0];
      const bool poisoned = seg_poison != 0ull && (row_mask() & seg_poison) != 0ull;
      const int node = R / a.g;  // the row's tree node
      const int64_t node_row = static_cast<int64_t>(sg.b) * a.R + node;
      // l_run = 0: the row saw no key here (the part drops out of the merge);
      // a non-finite l_run (a non-finite score) stays non-finite
      const float inv_l = l_run == 0.f ? 0.f : 1.f / l_run;
      const float lse_row = l_run == 0.f ? -INFINITY : m_run + __log2f(l_run);
      const int h = sg.hkv * a.g + (R - node * a.g);
      const int64_t out_row = node_row * a.Hq + h;
      if (whole) {
        // ---- the whole unit is in this segment: write the rows
        if (warp_valid) {
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(tO + q * 32, ov);
            tmem_wait_ld();
            if (valid) {
              uint4 *dst = reinterpret_cast<uint4 *>(a.out + out_row * D + q * 32);
#pragma unroll
              for (int k = 0; k < 32; k += 8) {
                uint4 v;
                v.x = dts::pack_bf16x2(__uint_as_float(ov[k]) * inv_l, __uint_as_float(ov[k + 1]) * inv_l);
                v.y = dts::pack_bf16x2(__uint_as_float(ov[k + 2]) * inv_l, __uint_as_float(ov[k + 3]) * inv_l);
                v.z = dts::pack_bf16x2(__uint_as_float(ov[k + 4]) * inv_l, __uint_as_float(ov[k + 5]) * inv_l);
                v.w = dts::pack_bf16x2(__uint_as_float(ov[k + 6]) * inv_l, __uint_as_float(ov[k + 7]) * inv_l);
                if (poisoned) v = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
                dst[k / 8] = v;
              }
            }
          }
          if (valid) a.lse2[out_row] = lse_row;
        }
        tc_fence_before();
        mbar_arrive(&o_free[t]);
      } else {
        // ---- one of several segments: write the partial (the merge pass
        // combines the unit's partials)
        const int64_t slot_row = (static_cast<int64_t>(sg.unit) + blockIdx.x) * a.slot_rows + prow;
        if (warp_valid) {
          // The partial row is normalised and stored in bf16, like the
          // output: its extra rounding (2^-9 relative) sits far inside the
          // output's tolerance and halves the bytes every split unit writes
          // here and the merge pass reads back. Thread = row, and a row is 2 D
          // contiguous bytes: stored straight, every store would hit another
          // row, and the epilogue would run at the rate of partial-sector
          // writes. So each 8-lane group transposes its 8 rows x 8 units (8
          // bytes = 4 columns) of a 32-column chunk (three xor-butterfly
          // stages) and then writes one row's 64 contiguous bytes per store.
          const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
          const int grp = lane & ~7, cu = lane & 7;
          uint16_t *dst0 = a.o_part + (slot_row - cu) * D + 4 * cu;  // row grp + 0, this lane's unit
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t ov[32];
            tmem_ld32(tO + q * 32, ov);
            tmem_wait_ld();
            uint2 u[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              u[k].x = dts::pack_bf16x2(__uint_as_float(ov[4 * k]) * inv_l, __uint_as_float(ov[4 * k + 1]) * inv_l);
              u[k].y = dts::pack_bf16x2(__uint_as_float(ov[4 * k + 2]) * inv_l, __uint_as_float(ov[4 * k + 3]) * inv_l);
              if (poisoned) u[k] = make_uint2(0x7FC07FC0u, 0x7FC07FC0u);
            }
#pragma unroll
            for (int mi = 0; mi < 3; ++mi) {
              const int m = 4 >> mi;
              const bool hi = (lane & m) != 0;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (k & m) continue;
                const uint2 snd = hi ? u[k] : u[k | m];
                uint2 rcv;
                rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, m);
                rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, m);
                if (hi) u[k] = rcv;
                else u[k | m] = rcv;
              }
            }
            // this lane now holds unit cu of rows grp .. grp + 7
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if ((vmask >> (grp + r)) & 1u) *reinterpret_cast<uint2 *>(dst0 + r * D + q * 32) = u[r];
          }
          if (valid) a.lse_part[slot_row] = lse_row;
          if (!F8 && a.unit_cnt != nullptr) {
            // This warp's rows of the part are stored. The CTA's last warp to
            // get here counts the part for the unit, and the CTA that counts
            // a unit's last part merges the unit at the end of the pass.
            __threadfence();
            __syncwarp();
            if (lane == 0) {
              int nvw = 0;  // warps of the CTA with rows in this part
              for (int tt = 0; tt < sg.nt; ++tt)
                for (int ww = 0; ww < 4; ++ww)
                  nvw += (ww * 32 < a.rt && sg.pair * 2 * a.rt + tt * a.rt + ww * 32 < a.M) ? 1 : 0;
              // only the range's first and last segments can be parts
              const int k = sg.start + sg.lt0 == x0 ? 0 : 1;
              if (atomicAdd(&part_cnt[k], 1) == nvw - 1) {
                __threadfence();
                const Owners own{total, static_cast<int64_t>(gridDim.x), a.owners32 != 0};
                const int64_t c_first = own.of(sg.start), c_last = own.of(sg.start + sg.nkt - 1);
                int parts = 0;
                for (int64_t cc = c_first; cc <= c_last; ++cc) parts += own.owns(cc) ? 1 : 0;
                if (atomicAdd(&a.unit_cnt[sg.unit], 1) == parts - 1) {
                  __threadfence();
                  const int e = atomicAdd(&part_cnt[2], 1);
                  MergeEntry me;
                  me.c_first = c_first;
                  me.c_last = c_last;
                  me.unit = static_cast<uint32_t>(sg.unit);
                  me.pair = sg.pair;
                  me.b = sg.b;
                  me.hkv = sg.hkv;
                  me.P = sg.P;
                  me.pad = 0;
                  mlist[e] = me;
                }
              }
            }
            __syncwarp();
          }
        }
        tc_fence_before();
        mbar_arrive(&o_free[t]);
      }
      tcnt += nkt;
      ++scnt;
    }
    if (!ok) {
      // The MMA warp may be blocked in the sync of round `arrived`, which
      // this warp has not joined. The abort flag is already set (by this
      // warp's timeout or by the role whose flag made the wait give up), so
      // one more arrival ends that sync and the MMA warp stops there. Round
      // arrived - 1 went to the other barrier, so this arrival cannot land
      // in it.
      named_arrive(p_bar_id(t, arrived), p_bar_threads(t));
      dts::report(a.err, DTS_DEV_TIMEOUT);
    }
    if (!F8 && a.unit_cnt != nullptr) {
      // the units whose last part this CTA stored (at most two: only the
      // range's first and last segments are parts), merged from every part,
      // 8 rows per warp, once all eight softmax warps are past their last
      // epilogue
      named_sync(kMergeBarrier, 256);
      if (*abort_flag == 0) {
        MergeArgs ma{};
        ma.o_part = a.o_part;
        ma.lse_part = a.lse_part;
        ma.out = a.out;
        ma.lse2 = a.lse2;
        ma.R = a.R;
        ma.Hq = a.Hq;
        ma.g = a.g;
        ma.M = a.M;
        ma.rt = a.rt;
        ma.slot_rows = a.slot_rows;
        const Owners own{total, static_cast<int64_t>(gridDim.x), a.owners32 != 0};
        const int n = part_cnt[2];
        const int rbs = (a.slot_rows + 7) / 8;
        for (int e = 0; e < n; ++e) {
          const MergeEntry me = mlist[e];
          for (int rb = warp - 4; rb < rbs; rb += 8)
            merge_rows<D, true>(ma, me.unit, rb, me.pair, me.b, me.hkv, me.P, me.c_first, me.c_last, own,
                                       lane);
        }
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

// Without F8, one warp per 8 consecutive rows of a unit's slot (lane l holds
// columns [E l, E l + E), E = d/32): a unit whose key tiles all fell to one
// CTA was written by the tree pass; the others merge their parts' partial
// rows by their LSEs: O = sum_k 2^(lse_k - m) O_k / sum_k 2^(lse_k - m), lse
// = m + log2(sum_k 2^(lse_k - m)), m the largest lse_k. Parts go four at a
// time: lane = part * 8 + row reads one LSE and decides once whether its
// group owns tiles; the row loads of the four parts follow. Under F8 every
// unit comes here, one CTA per 64 rows of its slot: its parts cover the
// prefix only, and merge_block_f8 adds the rows' window keys as one more part.
template <int D, bool F8>
__global__ void __launch_bounds__(256) tree_merge_kernel(const __grid_constant__ MergeArgs a) {
  dts::grid_dep_wait();
  dts::grid_dep_launch_next();
  constexpr int kRows = F8 ? 64 : 8;  // rows of a CTA (F8) or of a warp
  const int lane = threadIdx.x & 31;
  const uint32_t wid = F8 ? blockIdx.x : (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t blocks_per_unit = static_cast<uint32_t>((a.slot_rows + kRows - 1) / kRows);
  const uint32_t unit = wid / blocks_per_unit;
  // units in the flat order of the tree pass: (row pair, request, KV head)
  const uint32_t per_pair = static_cast<uint32_t>(a.B * a.Hkv);
  if (unit >= per_pair * static_cast<uint32_t>(a.n_pairs)) return;
  const int rb = static_cast<int>(wid - unit * blocks_per_unit);
  const int pair = static_cast<int>(unit / per_pair);
  const int bh = static_cast<int>(unit - static_cast<uint32_t>(pair) * per_pair);
  const int b = bh / a.Hkv, hkv = bh - b * a.Hkv;
  const int P = a.prefix_len[b];
  if (P < 0 || P > a.max_prefix || static_cast<int64_t>(P) + (F8 ? a.Ww : a.W) > a.capacity)
    return;  // NaN rows from prep
  const int nkt = (P + a.W + 127) >> 7;  // key tiles of the unit in the tree pass (F8: prefix only)
  const Owners own{a.tiles_before[a.B] * a.n_pairs, a.grid, a.owners32 != 0};
  const int64_t start = pair * a.tiles_before[a.B] + a.tiles_before[b] + static_cast<int64_t>(hkv) * nkt;
  const int64_t c_first = nkt > 0 ? own.of(start) : 0, c_last = nkt > 0 ? own.of(start + nkt - 1) : -1;
  if constexpr (F8) {
    merge_block_f8(a, unit, rb, pair, b, hkv, P, c_first, c_last, own);
  } else {
    if (c_first == c_last) return;  // one part: the tree pass wrote these rows
    merge_rows<D>(a, unit, rb, pair, b, hkv, P, c_first, c_last, own, lane);
  }
}

// ============================================================================
// host side
// ============================================================================
// Test hook (dts_test_stall_attention): the wait budget of the tree pass and
// whether its producer issues nothing.
std::atomic<long long> g_test_wait_budget{dts::ptx::kWaitBudget};
std::atomic<int> g_test_stall{0};

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

// L2 promotion: 256-byte fetches suit rows of 256 bytes or more; a 128-byte
// row (one KV head of an E4M3 cache) takes 128-byte fetches, so that a fetch
// does not also bring in the next head's row, which another CTA reads later.
bool encode(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
            const cuuint32_t *box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
            CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  auto enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dtype, rank, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (d, Hkv, slots) of a paged cache; box (64, 1, rows_per_box) for
// bf16, (128, 1, rows_per_box) for E4M3 bytes: 128 bytes a row either way.
bool make_cache_map(CUtensorMap *map, const void *base, int d, int Hkv, int64_t num_slots, int rows_per_box,
                    bool f8) {
  const cuuint64_t esz = f8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_slots)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz, static_cast<cuuint64_t>(Hkv) * d * esz};
  cuuint32_t box[3] = {f8 ? 128u : 64u, 1, static_cast<cuuint32_t>(rows_per_box)};
  return encode(map, base, 3, dims, strides, box, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                f8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// 4-D view (d, g, Hkv, B*N) of the queries [B*N][Hq][d]; box (64, g, 1, npt)
// of bf16, or (128, g, 1, npt) of E4M3 bytes: one box holds the npt * g rows
// (node, head-in-group) of a row tile, in that order.
bool make_q_map(CUtensorMap *map, const void *base, int d, int g, int Hkv, int64_t nodes, int npt, bool f8) {
  const cuuint64_t esz = f8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(nodes)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * esz, static_cast<cuuint64_t>(g) * d * esz,
                           static_cast<cuuint64_t>(g) * Hkv * d * esz};
  cuuint32_t box[4] = {f8 ? 128u : 64u, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(npt)};
  return encode(map, base, 4, dims, strides, box, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

template <int D, bool F8>
int launch_prefix(const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tq, const PrefixArgs &a, int grid,
                  cudaStream_t s) {
  using S = PrefixShape<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(tree_prefix_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(S::kSmem));
  });
  if (attr_err != cudaSuccess) return DTS_ERR_CUDA;
  dts_host::launch_chained(tree_prefix_kernel<D, F8>, dim3(grid), dim3(S::kThreads), S::kSmem, s, tk, tv, tq, a);
  return dts_host::launch_status();
}

}  // namespace

extern "C" size_t dts_tree_window_attention_workspace(int B, int R, int W, int Hq, int Hkv, int d,
                                                      int64_t max_prefix) {
  if (B <= 0 || R < 1 || R > dts::kMaxNodes || W < 1 || W > dts::kMaxNodes || Hkv < 1 || Hq < Hkv ||
      Hq % Hkv != 0 || Hq / Hkv > 128 || (d != 64 && d != 128) || max_prefix < 0)
    return 0;
  return static_cast<size_t>(make_plan(B, R, Hq, Hkv, d).total);
}

extern "C" size_t dts_tree_verify_attention_workspace(int B, int N, int Hq, int Hkv, int d, int64_t max_prefix) {
  return dts_tree_window_attention_workspace(B, N, N, Hq, Hkv, d, max_prefix);
}

namespace {

// Both cache types: bf16 (f8 = false) or unscaled E4M3 bytes (f8 = true).
int window_attention(bool f8, const uint16_t *q, const void *k_cache, const void *v_cache, int64_t num_slots,
                     const int32_t *page_table, int max_pages, int page_size, const int32_t *prefix_len,
                     int64_t max_prefix, const uint64_t *mask, const int32_t *positions, float rope_theta, int B, int R,
                     int W, int Hq, int Hkv, int d, float softmax_scale, uint16_t *out, float *lse2, void *workspace,
                     size_t ws_bytes, int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || R < 1 || W < 1 || Hkv < 1 || Hq < 1 || max_pages < 1 || num_slots < 1 || max_prefix < 0)
    return DTS_ERR_INVALID;
  if (R > dts::kMaxNodes || W > dts::kMaxNodes || (d != 64 && d != 128)) return DTS_ERR_UNSUPPORTED;
  if (f8 && d != 128) return DTS_ERR_UNSUPPORTED;
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
  if (static_cast<int64_t>(B) * R * Hq >= (1ll << 31) / d) return DTS_ERR_UNSUPPORTED;
  const Plan plan = make_plan(B, R, Hq, Hkv, d);
  if (workspace == nullptr || ws_bytes < static_cast<size_t>(plan.total)) return DTS_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  uint16_t *o_part = reinterpret_cast<uint16_t *>(ws + plan.o_off);
  float *lse_part = reinterpret_cast<float *>(ws + plan.lse_off);
  int64_t *tiles_before = reinterpret_cast<int64_t *>(ws + plan.tb_off);
  int32_t *unit_cnt = reinterpret_cast<int32_t *>(ws + plan.cnt_off);
  uint16_t *q_rot = reinterpret_cast<uint16_t *>(ws + plan.q_off);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.f / sqrtf(static_cast<float>(d));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int page_shift = __builtin_ctz(static_cast<unsigned>(page_size));
  const int g = Hq / Hkv;

  // Units of at most 128 rows split over CTAs are merged by the tree pass
  // itself (the CTA that stores a unit's last part, with its eight softmax
  // warps) when every CTA has many key tiles: such a merge is short against
  // the pass, and the merge launch is saved. Larger units (several parts of
  // 256 rows) go to the merge pass, which spreads them over the whole GPU; so
  // do short passes, where the merge would lengthen the last CTAs, and every
  // unit under F8, whose window keys the merge pass adds.
  const int sms = dts_host::sm_count();
  const int grid = sms > 0 ? (sms < kMaxGrid ? sms : kMaxGrid) : 1;
  const int64_t tiles_bound =
      static_cast<int64_t>(B) * Hkv * plan.n_pairs * ((max_prefix + (f8 ? 0 : W) + 127) / 128);
  const bool merge_in_pass = !f8 && plan.slot_rows <= 128 && tiles_bound >= 64ll * grid;

  // 0. prep: rotated queries, NaN rows for bad prefix lengths
  {
    PrepArgs ra;
    ra.q = q;
    ra.positions = positions;
    ra.prefix_len = prefix_len;
    ra.q_rot = q_rot;
    ra.out = out;
    ra.lse2 = lse2;
    ra.err = err_dev;
    ra.max_prefix = max_prefix;
    ra.capacity = static_cast<int64_t>(max_pages) << page_shift;
    ra.rows = B * R;
    ra.R = R;
    ra.W = W;
    ra.Hq = Hq;
    ra.heads_per_thread = (Hq % 4 == 0) ? 4 : (Hq % 2 == 0) ? 2 : 1;
    ra.to_e4m3 = f8 ? 1 : 0;
    ra.unit_cnt = merge_in_pass ? unit_cnt : nullptr;
    ra.units = plan.units;
    if (positions != nullptr) dts_host::make_rope_freqs(rope_theta, d, &ra.freqs);
    const int64_t items = static_cast<int64_t>(B) * R * (Hq / ra.heads_per_thread) * (d / 16);
    const int blocks = static_cast<int>((items + 255) / 256);
    if (d == 128) dts_host::launch_chained(attn_prep_kernel<128>, dim3(blocks), dim3(256), 0, s, ra);
    else dts_host::launch_chained(attn_prep_kernel<64>, dim3(blocks), dim3(256), 0, s, ra);
    if (dts_host::launch_status() != DTS_OK) return DTS_ERR_CUDA;
  }
  const uint16_t *q_eff = (positions != nullptr || f8) ? q_rot : q;

  // 1. tree attention, one CTA per SM
  CUtensorMap tk, tv, tq;
  const int rpb = page_size < 128 ? page_size : 128;
  if (!make_cache_map(&tk, k_cache, d, Hkv, num_slots, rpb, f8) ||
      !make_cache_map(&tv, v_cache, d, Hkv, num_slots, rpb, f8) ||
      !make_q_map(&tq, q_eff, d, g, Hkv, static_cast<int64_t>(B) * R, plan.npt, f8))
    return DTS_ERR_CUDA;
  PrefixArgs pa;
  pa.page_table = page_table;
  pa.prefix_len = prefix_len;
  pa.mask = mask;
  pa.o_part = o_part;
  pa.lse_part = lse_part;
  pa.tiles_before = tiles_before;
  pa.out = out;
  pa.lse2 = lse2;
  pa.err = err_dev;
  pa.num_slots = num_slots;
  pa.max_prefix = max_prefix;
  pa.B = B;
  pa.R = R;
  pa.W = f8 ? 0 : W;  // F8: the tree pass covers the prefix; the merge pass adds the window
  pa.Hq = Hq;
  pa.Hkv = Hkv;
  pa.g = g;
  pa.M = R * g;
  pa.rt = plan.rt;
  pa.npt = plan.npt;
  pa.n_pairs = plan.n_pairs;
  pa.slot_rows = plan.slot_rows;
  pa.max_pages = max_pages;
  pa.page_shift = page_shift;
  pa.scale_log2 = scale * kLog2e;
  pa.wait_budget = g_test_wait_budget.load(std::memory_order_relaxed);
  pa.stall = g_test_stall.load(std::memory_order_relaxed);
  pa.unit_cnt = merge_in_pass ? unit_cnt : nullptr;
  int owners32 = 0;
  {
    // the largest possible tile total, times the groups, against 2^32
    const int64_t max_tiles = static_cast<int64_t>(B) * Hkv * plan.n_pairs * ((max_prefix + pa.W + 127) / 128);
    owners32 = static_cast<double>(max_tiles + 1) * grid < 4294967296.0 ? 1 : 0;
  }
  pa.owners32 = owners32;
  const int st = f8          ? launch_prefix<128, true>(tk, tv, tq, pa, grid, s)
                 : d == 128 ? launch_prefix<128, false>(tk, tv, tq, pa, grid, s)
                            : launch_prefix<64, false>(tk, tv, tq, pa, grid, s);
  if (st != DTS_OK) return st;
  if (merge_in_pass) return DTS_OK;

  // 2. merge pass: units whose key tiles went to more than one CTA (F8:
  // every unit, with its rows' window keys)
  MergeArgs ma;
  ma.o_part = o_part;
  ma.lse_part = lse_part;
  ma.tiles_before = tiles_before;
  ma.prefix_len = prefix_len;
  ma.out = out;
  ma.lse2 = lse2;
  ma.max_prefix = max_prefix;
  ma.capacity = static_cast<int64_t>(max_pages) << page_shift;
  ma.B = B;
  ma.R = R;
  ma.W = pa.W;
  ma.Ww = W;
  ma.mask = mask;
  ma.k8 = static_cast<const uint8_t *>(k_cache);
  ma.v8 = static_cast<const uint8_t *>(v_cache);
  ma.page_table = page_table;
  ma.err = err_dev;
  ma.num_slots = num_slots;
  ma.max_pages = max_pages;
  ma.page_shift = page_shift;
  ma.scale_log2 = scale * kLog2e;
  ma.Hq = Hq;
  ma.Hkv = Hkv;
  ma.g = g;
  ma.M = R * g;
  ma.rt = plan.rt;
  ma.n_pairs = plan.n_pairs;
  ma.slot_rows = plan.slot_rows;
  ma.grid = grid;
  ma.owners32 = owners32;
  // (F8: one CTA of 256 threads per 64 rows of a unit; else one warp per 8 rows)
  const int64_t warps = plan.units * ((plan.slot_rows + 7) / 8);
  const int blocks = f8 ? static_cast<int>(plan.units * ((plan.slot_rows + 63) / 64))
                        : static_cast<int>((warps * 32 + 255) / 256);
  if (f8) dts_host::launch_chained(tree_merge_kernel<128, true>, dim3(blocks), dim3(256), 0, s, ma);
  else if (d == 128) dts_host::launch_chained(tree_merge_kernel<128, false>, dim3(blocks), dim3(256), 0, s, ma);
  else dts_host::launch_chained(tree_merge_kernel<64, false>, dim3(blocks), dim3(256), 0, s, ma);
  return dts_host::launch_status();
}

}  // namespace

extern "C" int dts_tree_window_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                         int64_t num_slots, const int32_t *page_table, int max_pages,
                                         int page_size, const int32_t *prefix_len, int64_t max_prefix,
                                         const uint64_t *mask, const int32_t *positions, float rope_theta,
                                         int B, int R, int W, int Hq, int Hkv, int d, float softmax_scale,
                                         uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                         int32_t *err_dev, dts_stream_t stream) {
  return window_attention(false, q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                          max_prefix, mask, positions, rope_theta, B, R, W, Hq, Hkv, d, softmax_scale, out, lse2,
                          workspace, ws_bytes, err_dev, stream);
}

extern "C" int dts_tree_window_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                             int64_t num_slots, const int32_t *page_table, int max_pages,
                                             int page_size, const int32_t *prefix_len, int64_t max_prefix,
                                             const uint64_t *mask, const int32_t *positions, float rope_theta,
                                             int B, int R, int W, int Hq, int Hkv, int d, float softmax_scale,
                                             uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                             int32_t *err_dev, dts_stream_t stream) {
  return window_attention(true, q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                          max_prefix, mask, positions, rope_theta, B, R, W, Hq, Hkv, d, softmax_scale, out, lse2,
                          workspace, ws_bytes, err_dev, stream);
}

extern "C" int dts_tree_verify_attention_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                             int64_t num_slots, const int32_t *page_table, int max_pages,
                                             int page_size, const int32_t *prefix_len, int64_t max_prefix,
                                             const uint64_t *mask, const int32_t *positions, float rope_theta,
                                             int B, int N, int Hq, int Hkv, int d, float softmax_scale,
                                             uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                             int32_t *err_dev, dts_stream_t stream) {
  return window_attention(true, q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                          max_prefix, mask, positions, rope_theta, B, N, N, Hq, Hkv, d, softmax_scale, out, lse2,
                          workspace, ws_bytes, err_dev, stream);
}

extern "C" int dts_tree_verify_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                         int64_t num_slots, const int32_t *page_table, int max_pages,
                                         int page_size, const int32_t *prefix_len, int64_t max_prefix,
                                         const uint64_t *mask, const int32_t *positions, float rope_theta,
                                         int B, int N, int Hq, int Hkv, int d, float softmax_scale,
                                         uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                         int32_t *err_dev, dts_stream_t stream) {
  // verify: the N tree nodes are both the query rows and the window keys
  return dts_tree_window_attention(q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                                   max_prefix, mask, positions, rope_theta, B, N, N, Hq, Hkv, d, softmax_scale, out,
                                   lse2, workspace, ws_bytes, err_dev, stream);
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
struct StaticWsEntry {
  unsigned long long ctx_id;  // the context the address belongs to
  void *ptr;
};
StaticWsEntry g_static_ws[kMaxDevices] = {};

// Identity of the calling thread's current context. A device reset ends the
// primary context and a later call runs in a new one, with a new id, where the
// array has been loaded again at a possibly different address.
bool current_context_id(unsigned long long *id) {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
    return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_workspace in the current device's context. The
// host-side name of the array is only a stand-in; its device address has to
// be asked for once per device and context, with that device current.
void *static_workspace(int *status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = DTS_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_static_ws_mutex);
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  StaticWsEntry &e = g_static_ws[dev];
  if (e.ptr == nullptr || !have_ctx || e.ctx_id != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) {
      *status = DTS_ERR_CUDA;
      return nullptr;
    }
    // the lookup creates the context if there was none yet: key the entry on it
    unsigned long long ctx_after = 0;
    e.ptr = p;
    e.ctx_id = current_context_id(&ctx_after) ? ctx_after : 0;
  }
  *status = DTS_OK;
  return e.ptr;
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
  // Shapes, pointers and B = 0 are checked by the regular entry point, so
  // both calls answer the same arguments alike. Given no workspace it launches
  // nothing and returns the argument error, DTS_OK for B = 0, or (arguments
  // valid) DTS_ERR_WORKSPACE; only then is the static array looked up.
  const int checked = dts_tree_verify_attention(q, k_cache, v_cache, num_slots, page_table, max_pages, page_size,
                                                prefix_len, max_prefix, mask, positions, rope_theta, B, N, Hq, Hkv,
                                                d, softmax_scale, out, lse2, nullptr, 0, err_dev, stream);
  if (checked != DTS_ERR_WORKSPACE) return checked;
  if (dts_tree_verify_attention_workspace(B, N, Hq, Hkv, d, max_prefix) > kStaticWorkspaceBytes)
    return DTS_ERR_WORKSPACE;
  int status = DTS_OK;
  void *ws = static_workspace(&status);
  if (ws == nullptr) return status;
  // No part of the workspace needs to start at zero: every byte a call reads
  // was written earlier in the same call.
  return dts_tree_verify_attention(q, k_cache, v_cache, num_slots, page_table, max_pages, page_size, prefix_len,
                                   max_prefix, mask, positions, rope_theta, B, N, Hq, Hkv, d, softmax_scale, out,
                                   lse2, ws, kStaticWorkspaceBytes, err_dev, stream);
}

// Test hook: see include/dts.h.
extern "C" int dts_test_stall_attention(int stall, long long wait_budget_cycles) {
  if (stall != 0 && stall != 1) return DTS_ERR_INVALID;
  if (wait_budget_cycles < (1ll << 16) || wait_budget_cycles > dts::ptx::kWaitBudget) return DTS_ERR_INVALID;
  g_test_stall.store(stall, std::memory_order_relaxed);
  g_test_wait_budget.store(stall ? wait_budget_cycles : dts::ptx::kWaitBudget, std::memory_order_relaxed);
  return DTS_OK;
}
