// The window K/V write of one node by one warp, shared by the window write
// kernel and the fused verify prologue. [TS] "Position follows depth, slot
// follows node index": node i's key, rotated at vc + depth[i], and its value
// go to the slot of logical position prefix_len[b] + i. Lane l holds the
// rotate-half pairs (2l, 2l+1 | d/2+2l, d/2+2l+1) for d = 128, or (l | d/2+l)
// for d = 64. An FP8 cache ([TS] "One tree attention", FP8 paragraph: E4M3,
// unscaled) stores the same values cast to E4M3: the rotated key as rounded
// to bf16, and the value, each rounded to nearest even and saturated at +-448.
#pragma once

#include "common.cuh"

namespace dts {

struct WindowKvArgs {
  const uint16_t *k_new;
  const uint16_t *v_new;
  const int32_t *positions;
  const int32_t *page_table;
  const int32_t *prefix_len;
  void *k_cache;  // bf16, or E4M3 bytes (F8)
  void *v_cache;
  int64_t *write_locations;
  int32_t *err;
  int64_t num_slots;
  int max_pages, page_shift, B, N, Hkv;
  dts::RopeFreqs freqs;
};

// One warp writes node `node` (= b * N + i), rotated at `pos`: the RoPE
// angles depend on the node only, so they are computed once and applied to
// all its KV heads; every head's K and V loads are issued before the
// page-table lookup.
template <int D, bool F8>
__device__ __forceinline__ void write_node_kv(const WindowKvArgs &a, int node, int pos, int lane) {
  static_assert(!F8 || D == 128, "the FP8 cache takes d = 128");
  constexpr int kMaxHeads = 16;  // heads held in registers per pass
  const int b = node / a.N;
  const int i = node - b * a.N;
  const int P = a.prefix_len[b];
  const int ps = 1 << a.page_shift;
  const int64_t logical = static_cast<int64_t>(P) + i;
  const int64_t page = logical >> a.page_shift;
  const bool page_ok = P >= 0 && page < a.max_pages;
  const int pid = page_ok ? a.page_table[static_cast<int64_t>(b) * a.max_pages + page] : -1;
  for (int h0 = 0; h0 < a.Hkv; h0 += kMaxHeads) {
    const int nh = min(kMaxHeads, a.Hkv - h0);
    uint32_t k1[kMaxHeads], k2[kMaxHeads];
    uint2 v[kMaxHeads];
#pragma unroll
    for (int u = 0; u < kMaxHeads; ++u) {
      if (u >= nh) break;
      const uint16_t *kin = a.k_new + (static_cast<int64_t>(node) * a.Hkv + h0 + u) * D;
      const uint16_t *vin = a.v_new + (static_cast<int64_t>(node) * a.Hkv + h0 + u) * D;
      if constexpr (D == 128) {
        k1[u] = reinterpret_cast<const uint32_t *>(kin)[lane];       // elems 2l, 2l+1
        k2[u] = reinterpret_cast<const uint32_t *>(kin + 64)[lane];  // elems 64+2l, 64+2l+1
        v[u] = reinterpret_cast<const uint2 *>(vin)[lane];
      } else {
        k1[u] = kin[lane];
        k2[u] = kin[32 + lane];
        v[u].x = reinterpret_cast<const uint32_t *>(vin)[lane];
        v[u].y = 0;
      }
    }
    const int64_t slot = static_cast<int64_t>(pid) * ps + (logical & (ps - 1));
    if (pid < 0 || slot >= a.num_slots) {
      if (lane == 0 && h0 == 0) {
        dts::report(a.err, DTS_DEV_BAD_SLOT);
        if (a.write_locations) a.write_locations[node] = -1;
      }
      return;
    }
    if (lane == 0 && h0 == 0 && a.write_locations) a.write_locations[node] = slot;
    if constexpr (D == 128) {
      const int k0 = 2 * lane;
      float s0, c0, s1, c1;
      dts::rope_sincos(pos, a.freqs.w[k0], &s0, &c0);
      dts::rope_sincos(pos, a.freqs.w[k0 + 1], &s1, &c1);
#pragma unroll
      for (int u = 0; u < kMaxHeads; ++u) {
        if (u >= nh) break;
        const int64_t row = (slot * a.Hkv + h0 + u) * D;
        const float a0 = dts::bf16_lo(k1[u]), a1 = dts::bf16_hi(k1[u]);
        const float b0 = dts::bf16_lo(k2[u]), b1 = dts::bf16_hi(k2[u]);
        const uint32_t r1 = dts::pack_bf16x2(a0 * c0 - b0 * s0, a1 * c1 - b1 * s1);
        const uint32_t r2 = dts::pack_bf16x2(b0 * c0 + a0 * s0, b1 * c1 + a1 * s1);
        if constexpr (F8) {
          uint8_t *kout = static_cast<uint8_t *>(a.k_cache) + row;
          uint8_t *vout = static_cast<uint8_t *>(a.v_cache) + row;
          reinterpret_cast<uint16_t *>(kout)[lane] =
              static_cast<uint16_t>(dts::f32x2_to_e4m3x2(dts::bf16_lo(r1), dts::bf16_hi(r1)));
          reinterpret_cast<uint16_t *>(kout + 64)[lane] =
              static_cast<uint16_t>(dts::f32x2_to_e4m3x2(dts::bf16_lo(r2), dts::bf16_hi(r2)));
          const uint32_t v01 = dts::f32x2_to_e4m3x2(dts::bf16_lo(v[u].x), dts::bf16_hi(v[u].x));
          const uint32_t v23 = dts::f32x2_to_e4m3x2(dts::bf16_lo(v[u].y), dts::bf16_hi(v[u].y));
          reinterpret_cast<uint32_t *>(vout)[lane] = v01 | (v23 << 16);
        } else {
          uint16_t *kout = static_cast<uint16_t *>(a.k_cache) + row;
          uint16_t *vout = static_cast<uint16_t *>(a.v_cache) + row;
          reinterpret_cast<uint32_t *>(kout)[lane] = r1;
          reinterpret_cast<uint32_t *>(kout + 64)[lane] = r2;
          reinterpret_cast<uint2 *>(vout)[lane] = v[u];
        }
      }
    } else if constexpr (!F8) {
      float s0, c0;
      dts::rope_sincos(pos, a.freqs.w[lane], &s0, &c0);
#pragma unroll
      for (int u = 0; u < kMaxHeads; ++u) {
        if (u >= nh) break;
        uint16_t *kout = static_cast<uint16_t *>(a.k_cache) + (slot * a.Hkv + h0 + u) * D;
        uint16_t *vout = static_cast<uint16_t *>(a.v_cache) + (slot * a.Hkv + h0 + u) * D;
        const float a0 = __uint_as_float(k1[u] << 16);
        const float b0 = __uint_as_float(k2[u] << 16);
        const uint32_t r = dts::pack_bf16x2(a0 * c0 - b0 * s0, b0 * c0 + a0 * s0);
        kout[lane] = static_cast<uint16_t>(r & 0xFFFFu);
        kout[32 + lane] = static_cast<uint16_t>(r >> 16);
        reinterpret_cast<uint32_t *>(vout)[lane] = v[u].x;
      }
    }
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(256) write_window_kv_kernel(const __grid_constant__ WindowKvArgs a) {
  const int node = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // b * N + i
  if (node >= a.B * a.N) return;
  write_node_kv<D, F8>(a, node, a.positions[node], threadIdx.x & 31);
}

}  // namespace dts
