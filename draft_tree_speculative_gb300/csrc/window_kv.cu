// Window K/V write entry points (bf16 and E4M3 caches): one warp per node,
// the per-node write in window_kv.cuh.
#include "window_kv.cuh"

namespace {

using dts::WindowKvArgs;
using dts::write_window_kv_kernel;

int write_window_kv(bool f8, const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                    const int32_t *page_table, int max_pages, int page_size, const int32_t *prefix_len, int B, int N,
                    int Hkv, int d, int64_t num_slots, float rope_theta, void *k_cache, void *v_cache,
                    int64_t *write_locations, int32_t *err_dev, dts_stream_t stream) {
  if (B < 0 || N < 1 || Hkv < 1 || max_pages < 1 || num_slots < 1) return DTS_ERR_INVALID;
  if (N > dts::kMaxNodes || (d != 64 && d != 128)) return DTS_ERR_UNSUPPORTED;
  if (f8 && d != 128) return DTS_ERR_UNSUPPORTED;
  if (page_size < 8 || page_size > 4096 || (page_size & (page_size - 1)) != 0) return DTS_ERR_UNSUPPORTED;
  if (!(rope_theta > 0.f)) return DTS_ERR_INVALID;
  if (B == 0) return DTS_OK;
  if (!k_new || !v_new || !positions || !page_table || !prefix_len || !k_cache || !v_cache)
    return DTS_ERR_INVALID;
  const uintptr_t al = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
  if (al & 7) return DTS_ERR_INVALID;  // (an E4M3 row of 128 bytes keeps every store aligned too)
  WindowKvArgs a;
  a.k_new = k_new;
  a.v_new = v_new;
  a.positions = positions;
  a.page_table = page_table;
  a.prefix_len = prefix_len;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.write_locations = write_locations;
  a.err = err_dev;
  a.num_slots = num_slots;
  a.max_pages = max_pages;
  a.page_shift = __builtin_ctz(static_cast<unsigned>(page_size));
  a.B = B;
  a.N = N;
  a.Hkv = Hkv;
  dts_host::make_rope_freqs(rope_theta, d, &a.freqs);
  const int64_t warps = static_cast<int64_t>(B) * N;
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (f8) write_window_kv_kernel<128, true><<<blocks, 256, 0, s>>>(a);
  else if (d == 128) write_window_kv_kernel<128, false><<<blocks, 256, 0, s>>>(a);
  else write_window_kv_kernel<64, false><<<blocks, 256, 0, s>>>(a);
  return dts_host::launch_status();
}

}  // namespace

extern "C" int dts_write_window_kv(const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                                   const int32_t *page_table, int max_pages, int page_size,
                                   const int32_t *prefix_len, int B, int N, int Hkv, int d,
                                   int64_t num_slots, float rope_theta, uint16_t *k_cache,
                                   uint16_t *v_cache, int64_t *write_locations, int32_t *err_dev,
                                   dts_stream_t stream) {
  return write_window_kv(false, k_new, v_new, positions, page_table, max_pages, page_size, prefix_len, B, N, Hkv, d,
                         num_slots, rope_theta, k_cache, v_cache, write_locations, err_dev, stream);
}

extern "C" int dts_write_window_kv_fp8(const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                                       const int32_t *page_table, int max_pages, int page_size,
                                       const int32_t *prefix_len, int B, int N, int Hkv, int d,
                                       int64_t num_slots, float rope_theta, uint8_t *k_cache,
                                       uint8_t *v_cache, int64_t *write_locations, int32_t *err_dev,
                                       dts_stream_t stream) {
  return write_window_kv(true, k_new, v_new, positions, page_table, max_pages, page_size, prefix_len, B, N, Hkv, d,
                         num_slots, rope_theta, k_cache, v_cache, write_locations, err_dev, stream);
}
