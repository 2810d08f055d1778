/*
 * dts.h - C ABI of the target-verify step of draft-tree speculative decoding,
 * built for GB300 (sm_103a).
 *
 * A verify step runs the N <= 64 nodes of one draft tree per request through
 * one target forward. This library provides that step's data-parallel path:
 *
 *   dts_build_tree_mask         parents/depth -> 64-bit ancestor masks,
 *                               positions vc + depth, first-child/next-sibling
 *   dts_write_window_kv         RoPE'd window K and V into the paged cache
 *   dts_tree_verify_attention   every row attends the committed prefix plus
 *                               its own ancestors; out + base-2 LSE
 *   dts_tree_window_attention   the same over R rows and a W-key masked window
 *                               (draft lanes: R = K rows, W = (S - 1) * K keys)
 *   dts_*_fp8                   the window write and both attentions over an
 *                               unscaled FP8-E4M3 KV cache
 *   dts_verify_tree_greedy      greedy walk -> accept_len, packed path, tokens
 *   dts_target_argmax           the target's argmax per verify row (and
 *   dts_verify_tree_greedy_logits  that argmax fed straight into the walk)
 *   dts_sample_draws            sampled draws, Gumbel-max keyed by position (and
 *   dts_verify_tree_sampled     the walk over them)
 *   dts_compact_window_rows     the path's KV rows -> the window's front slots
 *   dts_compact_rows            the path's hidden rows -> the front; positions
 *                               back to vc + i
 *
 * Sources (web pages, cited by title and section):
 *   [TS] "Draft-tree speculation" (tokenspeed design notes)
 *   [AK] "EAGLE Tree Attention candidate layout, positions and visibility"
 *        (DeepSeek-V4 tree-attention source analysis)
 *   [MI] "Medusa, EAGLE-1/2/3, MTP, and tree attention" (chapter 6.4)
 *   [DD] "From Greedy to Sampling: The Architecture of Choice in DDTree
 *        Speculative Decoding"
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller, unless the
 *     comment says otherwise. The library never allocates, frees or keeps a
 *     pointer after the call returns.
 *   - bf16 tensors are passed as uint16_t storage (the raw bf16 bits).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronises, so the calls can be
 *     captured in a CUDA graph.
 *   - The return value is a host-side status (DTS_OK or a negative
 *     DTS_ERR_*), found before anything is launched, or DTS_ERR_CUDA if a
 *     launch failed.
 *   - Data errors that only the device can see (a bad parent index, a page id
 *     out of range, ...) never trap: the kernel writes a DTS_DEV_* code to
 *     *err_dev (an int32 in device memory; the first error wins, so the caller
 *     zeroes it before a step and reads it when convenient) and skips the bad
 *     item. err_dev may be NULL, in which case such errors go unreported.
 */
#ifndef DTS_H
#define DTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *dts_stream_t; /* == cudaStream_t */

/* host-side status codes */
#define DTS_OK 0
#define DTS_ERR_INVALID (-1)     /* null pointer, bad shape or alignment */
#define DTS_ERR_UNSUPPORTED (-2) /* N > 64, d not 64/128, ... */
#define DTS_ERR_WORKSPACE (-3)   /* workspace missing or too small */
#define DTS_ERR_CUDA (-4)        /* a kernel launch or driver call failed */

/* device-detected data errors written to *err_dev */
#define DTS_DEV_OK 0
#define DTS_DEV_BAD_PARENT 1   /* parents[0] != -1, or not 0 <= parents[i] < i */
#define DTS_DEV_BAD_DEPTH 2    /* depth[0] != 0, or depth[i] != depth[parent]+1 */
#define DTS_DEV_BAD_LINK 3     /* next_token/next_sibling out of range or cyclic */
#define DTS_DEV_BAD_SLOT 4     /* page id, slot or prefix length out of range */
#define DTS_DEV_BAD_PATH 5     /* accept_len / accepted_path not a valid packed path */
#define DTS_DEV_BAD_BUFFER 6   /* a KV buffer entry is misaligned or partly overlaps another */
#define DTS_DEV_TIMEOUT 7      /* a bounded wait inside a kernel gave up */

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int dts_version(void);

/* Readable text for a DTS_* status or a DTS_DEV_* code. Static strings. */
const char *dts_status_string(int status);
const char *dts_device_error_string(int code);

/*
 * dts_build_tree_mask - validate B trees and derive what the verify forward
 * and the walk need.
 *
 * Defined by [TS] "One tree attention" (one 64-bit ancestor mask per row),
 * "Position follows depth, slot follows node index" (position vc + depth[i]),
 * [AK] section one (a row sees the prefix, itself and its ancestors) and [MI]
 * "Flattening, and the two link arrays" (first-child / next-sibling).
 *
 *   parents   int32 [B][N]  parents[b][0] = -1 (the root), 0 <= parents[b][i] < i
 *   depth     int32 [B][N]  depth[b][0] = 0, depth[b][i] = depth[b][parents[b][i]] + 1
 *   vc        int32 [B]     committed prefix length of each request
 *   mask      u64   [B][N]  out: bit j of mask[b][i] set iff j == i or j is an
 *                           ancestor of i
 *   positions int32 [B][N]  out: vc[b] + depth[b][i]
 *   next_token   int32 [B][N] out: lowest-index child of i, or -1
 *   next_sibling int32 [B][N] out: next-higher-index child of i's parent, or -1
 *
 * 1 <= N <= 64, B >= 0 (B = 0 launches nothing). A request whose tree is
 * invalid gets DTS_DEV_BAD_PARENT or DTS_DEV_BAD_DEPTH in *err_dev and all of
 * its outputs set to 0 / -1 (mask 0, positions vc, links -1).
 */
int dts_build_tree_mask(const int32_t *parents, const int32_t *depth, const int32_t *vc,
                        int B, int N, uint64_t *mask, int32_t *positions,
                        int32_t *next_token, int32_t *next_sibling, int32_t *err_dev,
                        dts_stream_t stream);

/*
 * dts_write_window_kv - store the window's K (rotated) and V in the paged cache.
 *
 * Defined by [TS] "Position follows depth, slot follows node index": node i's
 * K/V go to the slot of logical position vc + i (slot follows node index),
 * and K is rotated at positions[b][i] = vc + depth[i] (position follows depth).
 * RoPE reading: rotate-half pairs (x_k, x_{k+d/2}), angle pos * theta^(-2k/d).
 *
 *   k_new, v_new  bf16 [B*N][Hkv][d]   the window's new keys (not rotated) and values
 *   positions     int32 [B][N]         RoPE position of each node
 *   page_table    int32 [B][max_pages] physical page of each logical page
 *   prefix_len    int32 [B]            P_b = vc: node i lives at logical position P_b + i
 *   k_cache, v_cache bf16 [num_slots][Hkv][d], slot = page * page_size + offset
 *   write_locations int64 [B*N]        optional out (NULL = skip): the slot of each node
 *
 * d in {64, 128}; page_size a power of two in [8, 4096]; Hkv >= 1.
 * A page id or slot out of range gives DTS_DEV_BAD_SLOT and skips that node.
 */
int dts_write_window_kv(const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                        const int32_t *page_table, int max_pages, int page_size,
                        const int32_t *prefix_len, int B, int N, int Hkv, int d,
                        int64_t num_slots, float rope_theta, uint16_t *k_cache,
                        uint16_t *v_cache, int64_t *write_locations, int32_t *err_dev,
                        dts_stream_t stream);

/*
 * dts_tree_verify_attention_workspace - bytes of device workspace that
 * dts_tree_verify_attention needs for these sizes (0 never happens for B > 0).
 * max_prefix is an upper bound on every prefix_len[b]. Host-only; no CUDA call.
 */
size_t dts_tree_verify_attention_workspace(int B, int N, int Hq, int Hkv, int d,
                                           int64_t max_prefix);

/*
 * dts_tree_verify_attention - attention of the N verify rows of each request.
 *
 * Defined by [TS] "One tree attention": every row sees the committed prefix,
 * and the 64-bit ancestor mask applies only to the last W = N keys (the
 * window); the result carries a base-2 log-sum-exp. [AK] section one: row v
 * must equal Target(prefix + path(root -> v)). [AK] section four: partial
 * results over disjoint key sets merge by their log-sum-exps.
 *
 *   q          bf16 [B*N][Hq][d]       queries; rotated here at positions[b][i]
 *                                      unless positions is NULL (then taken as
 *                                      already rotated)
 *   k_cache, v_cache bf16 [num_slots][Hkv][d]  paged cache; prefix keys already
 *                                      rotated; window keys written by
 *                                      dts_write_window_kv
 *   page_table int32 [B][max_pages]
 *   prefix_len int32 [B]               P_b; window node j is at logical position P_b + j
 *   max_prefix host int64              upper bound on every P_b (plans the KV split)
 *   mask       u64 [B][N]              from dts_build_tree_mask
 *   positions  int32 [B][N] or NULL
 *   softmax_scale  0 -> 1/sqrt(d)
 *   out        bf16 [B*N][Hq][d]       out: normalised attention output
 *   lse2       fp32 [B*N][Hq]          out: log2(sum_j exp(s_j)) over the row's keys
 *   workspace  device, >= dts_tree_verify_attention_workspace(...) bytes,
 *              16-byte aligned; its contents on entry do not matter
 *
 * Query head h reads KV head h / (Hq/Hkv). d in {64, 128}; Hq % Hkv == 0;
 * 1 <= N <= 64; page_size a power of two in [8, 4096]; cache and q base
 * addresses 16-byte aligned. Window keys that a row's mask does not select
 * count for nothing in that row: a non-finite K or V row of a window key
 * makes only the rows that see it non-finite, and slots past the window never
 * reach any row. A row whose mask is 0 and whose prefix is empty gets out = 0
 * and lse2 = -inf. A request whose prefix_len[b] is < 0, > max_prefix, or
 * puts the window past max_pages * page_size gets NaN rows and
 * DTS_DEV_BAD_SLOT; so does a page id outside the pool.
 * Launches three kernels on `stream` (query rotation, the tensor-core pass
 * over prefix and window keys, the merge of units split over CTAs), or two
 * when the tensor-core pass merges the split units itself (units of at most
 * 128 query rows on a long pass). The kernels are chained by programmatic
 * dependent launch, each waiting for its predecessor before it reads memory.
 */
int dts_tree_verify_attention(const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, int64_t num_slots,
                              const int32_t *page_table, int max_pages, int page_size,
                              const int32_t *prefix_len, int64_t max_prefix,
                              const uint64_t *mask, const int32_t *positions,
                              float rope_theta, int B, int N, int Hq, int Hkv, int d,
                              float softmax_scale, uint16_t *out, float *lse2,
                              void *workspace, size_t ws_bytes, int32_t *err_dev,
                              dts_stream_t stream);

/*
 * dts_tree_window_attention_workspace - bytes of device workspace that
 * dts_tree_window_attention needs (the same plan as
 * dts_tree_verify_attention_workspace with R query rows per request; W does
 * not enter it), or 0 if the shape is unsupported. Host-only.
 */
size_t dts_tree_window_attention_workspace(int B, int R, int W, int Hq, int Hkv, int d,
                                           int64_t max_prefix);

/*
 * dts_tree_window_attention - attention of R query rows per request over the
 * committed prefix plus a masked window of W keys (the general form of
 * dts_tree_verify_attention, which is this call with R = W = N).
 *
 * Defined by [TS] "One tree attention": every row sees the committed prefix,
 * and the 64-bit mask applies only to the last W keys; verify runs it with
 * R = W = N, draft lanes with R = K rows over the (S - 1) * K-key lane window.
 * [TS] "Draft lanes write the draft cache like any draft step": every lane row
 * sees the accepted frontier and, inside the window, only its ancestors'
 * slots (the lane mask); step s lane r writes slot frontier + (s - 1) * K + r.
 *
 *   q          bf16 [B*R][Hq][d]       row r of request b at b*R + r; rotated
 *                                      here at positions[b][r] unless
 *                                      positions is NULL
 *   k_cache, v_cache bf16 [num_slots][Hkv][d]  paged cache holding the prefix
 *                                      and the window, all keys already rotated
 *                                      at their own positions
 *   page_table, prefix_len, max_prefix as for dts_tree_verify_attention;
 *                                      window key j is at logical position P_b + j
 *   mask       u64 [B][R]              bit j: row r sees window key j (j < W)
 *   positions  int32 [B][R] or NULL
 *   out        bf16 [B*R][Hq][d]; lse2 fp32 [B*R][Hq]   outputs
 *   workspace  device, >= dts_tree_window_attention_workspace(...) bytes
 *
 * 1 <= R <= 64 and 1 <= W <= 64; every other constraint, output rule and
 * error is as for dts_tree_verify_attention (with W in place of N for the
 * window and R for the rows).
 */
int dts_tree_window_attention(const uint16_t *q, const uint16_t *k_cache,
                              const uint16_t *v_cache, int64_t num_slots,
                              const int32_t *page_table, int max_pages, int page_size,
                              const int32_t *prefix_len, int64_t max_prefix,
                              const uint64_t *mask, const int32_t *positions, float rope_theta,
                              int B, int R, int W, int Hq, int Hkv, int d, float softmax_scale,
                              uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                              int32_t *err_dev, dts_stream_t stream);

/*
 * FP8-E4M3 KV cache.
 *
 * Defined by [TS] "One tree attention", FP8 paragraph: an FP8 KV cache is
 * E4M3 and unscaled (a byte is the value itself), it changes none of the
 * structure, and the window's FP8 K/V are widened to the model dtype after
 * loading, with the unquantized query. Format: 1 sign bit, 4 exponent bits
 * (bias 7), 3 mantissa bits, S.1111.111 = NaN, no infinity, largest 448.
 *
 * dts_write_window_kv_fp8 - dts_write_window_kv into E4M3 caches
 * [num_slots][Hkv][d] (bytes). Stored values: the rotated key as rounded to
 * bf16, then cast to E4M3, and the value cast to E4M3; the cast rounds to
 * nearest even and saturates at +-448 (NaN stays NaN). d = 128 only
 * (DTS_ERR_UNSUPPORTED otherwise); every other argument, rule and error is
 * dts_write_window_kv's.
 *
 * dts_tree_window_attention_fp8 / dts_tree_verify_attention_fp8 -
 * dts_tree_window_attention / dts_tree_verify_attention over E4M3 caches
 * [num_slots][Hkv][d] (bytes, 16-byte aligned), with the same workspace
 * sizes (dts_tree_window_attention_workspace /
 * dts_tree_verify_attention_workspace). The query is rotated and rounded to
 * bf16 as for the bf16 cache (or taken as given when positions is NULL). The
 * prefix keys [0, P) are scored against that query cast to E4M3, as the
 * prefix decode over an FP8 cache does: S = Q K^T is one E4M3 tensor-core
 * product with fp32 accumulation, V is widened to f16 (exact), the softmax
 * weights enter P.V as f16 and accumulate in fp32. The window keys [P, P + W)
 * are scored against the unquantized bf16 query, with their K and V rows
 * widened exactly from E4M3 and fp32 arithmetic; the two parts then merge by
 * their log-sum-exps. d = 128 only (DTS_ERR_UNSUPPORTED otherwise); every
 * other argument, output rule and error is that of the bf16 call, a NaN byte
 * in a window key's V row standing for the non-finite V row there.
 */
int dts_write_window_kv_fp8(const uint16_t *k_new, const uint16_t *v_new, const int32_t *positions,
                            const int32_t *page_table, int max_pages, int page_size,
                            const int32_t *prefix_len, int B, int N, int Hkv, int d,
                            int64_t num_slots, float rope_theta, uint8_t *k_cache,
                            uint8_t *v_cache, int64_t *write_locations, int32_t *err_dev,
                            dts_stream_t stream);
int dts_tree_window_attention_fp8(const uint16_t *q, const uint8_t *k_cache,
                                  const uint8_t *v_cache, int64_t num_slots,
                                  const int32_t *page_table, int max_pages, int page_size,
                                  const int32_t *prefix_len, int64_t max_prefix,
                                  const uint64_t *mask, const int32_t *positions, float rope_theta,
                                  int B, int R, int W, int Hq, int Hkv, int d, float softmax_scale,
                                  uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                  int32_t *err_dev, dts_stream_t stream);
int dts_tree_verify_attention_fp8(const uint16_t *q, const uint8_t *k_cache,
                                  const uint8_t *v_cache, int64_t num_slots,
                                  const int32_t *page_table, int max_pages, int page_size,
                                  const int32_t *prefix_len, int64_t max_prefix,
                                  const uint64_t *mask, const int32_t *positions, float rope_theta,
                                  int B, int N, int Hq, int Hkv, int d, float softmax_scale,
                                  uint16_t *out, float *lse2, void *workspace, size_t ws_bytes,
                                  int32_t *err_dev, dts_stream_t stream);

/*
 * dts_tree_verify_attention_static_ws - dts_tree_verify_attention without a
 * caller-supplied workspace. The pages have no counterpart: this is a service
 * for callers that cannot allocate device memory, such as a process whose own
 * pool already holds the whole device, a plugin without access to its host's
 * allocator, or code that must not call cudaMalloc while it runs.
 *
 * Arguments and results are those of dts_tree_verify_attention, minus
 * workspace/ws_bytes. The scratch space is a fixed 64 MiB array in the
 * library's device image; every GPU that loads the library holds it until the
 * process exits. Shapes whose workspace (dts_tree_verify_attention_workspace)
 * exceeds 64 MiB get DTS_ERR_WORKSPACE and nothing runs.
 *
 * Arguments are validated exactly as dts_tree_verify_attention validates
 * them (B = 0 returns DTS_OK), before the array is touched.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it, keyed by the
 * current context: after a device reset the next call looks it up again in
 * the new context. Make the first call on a device (and the first after a
 * reset) before any stream capture. The call allocates and frees nothing.
 * All calls share the one array: calls whose work overlaps on the GPU (other
 * streams, other host threads) race and give wrong results, so serialise them.
 * Nothing in the array needs clearing between calls.
 */
int dts_tree_verify_attention_static_ws(const uint16_t *q, const uint16_t *k_cache,
                                        const uint16_t *v_cache, int64_t num_slots,
                                        const int32_t *page_table, int max_pages, int page_size,
                                        const int32_t *prefix_len, int64_t max_prefix,
                                        const uint64_t *mask, const int32_t *positions,
                                        float rope_theta, int B, int N, int Hq, int Hkv, int d,
                                        float softmax_scale, uint16_t *out, float *lse2,
                                        int32_t *err_dev, dts_stream_t stream);

/*
 * dts_verify_tree_greedy - greedy tree verification, one warp per request.
 *
 * Defined by [MI] "Walking the accepted path": from the root, descend to the
 * first child, scan the siblings for one whose draft token equals the
 * target's argmax at the parent, accept it and repeat; stop when no sibling
 * matches. [AK] section two: accept_len = correct drafts + 1; the accepted
 * outputs are the target argmax at each accepted node (the last is the bonus).
 * [TS] "The tree is a parameter of the chain path": the path is packed.
 *
 *   draft_tokens, target_argmax int32 [B][N]
 *   next_token, next_sibling    int32 [B][N]  the links (from dts_build_tree_mask),
 *                               or both NULL to derive children from parents
 *   parents                     int32 [B][N]  used only when the links are NULL
 *   accept_len       int32 [B]     out: number of accepted nodes, >= 1
 *   accepted_path    int32 [B][N]  out: accepted node ids (local), -1 padded
 *   accepted_tokens  int32 [B][N]  out: target_argmax at each accepted node, -1 padded
 *
 * Siblings are scanned in link order (ascending node index when the links come
 * from dts_build_tree_mask or from parents); the first match wins. A link out
 * of range or a cycle gives DTS_DEV_BAD_LINK and accept_len = 1.
 */
int dts_verify_tree_greedy(const int32_t *draft_tokens, const int32_t *target_argmax,
                           const int32_t *parents, const int32_t *next_token,
                           const int32_t *next_sibling, int B, int N, int32_t *accept_len,
                           int32_t *accepted_path, int32_t *accepted_tokens,
                           int32_t *err_dev, dts_stream_t stream);

/*
 * dts_target_argmax_workspace - bytes of scratch dts_target_argmax and
 * dts_verify_tree_greedy_logits need for `rows` rows of `vocab` logits
 * (8 bytes per row and 16384-logit chunk), or 0 for rows < 0 or vocab < 1.
 */
size_t dts_target_argmax_workspace(int64_t rows, int vocab);

/*
 * dts_target_argmax - the target's argmax at every verify row.
 *
 * Defined by [MI] "Walking the accepted path": the walk compares the draft
 * tokens with the target's argmax at each node's position, computed for all
 * nodes by the one verify forward; [MI], the worked (5, 4, 8) iteration, step
 * 5: the argmax over all rows, then the walk.
 *
 *   logits     float [rows][row_stride]  row r's vocab logits at r * row_stride
 *              (row_stride >= vocab, in elements; 4-byte aligned; rows that
 *              start on 16-byte boundaries are read as float4 words)
 *   argmax     int32 [rows]              out: index of the row's largest logit
 *   workspace  device scratch of dts_target_argmax_workspace(rows, vocab)
 *              bytes, 8-byte aligned, owned by the caller; nothing in it needs
 *              to start at zero, and it is free again when the call's work on
 *              `stream` has finished
 *
 * Ties go to the lowest index; a NaN counts as larger than any number (the
 * first NaN of a row wins); -0.0 equals +0.0. Returns DTS_ERR_INVALID for a
 * bad shape, pointer or alignment, DTS_ERR_WORKSPACE for a missing or small
 * workspace, DTS_ERR_UNSUPPORTED when rows x chunks reaches 2^31.
 */
int dts_target_argmax(const float *logits, int64_t rows, int vocab, int64_t row_stride,
                      int32_t *argmax, void *workspace, size_t ws_bytes, dts_stream_t stream);

/*
 * dts_verify_tree_greedy_logits - the target's argmax at every verify row
 * (dts_target_argmax over logits [B*N][row_stride], row b*N+i for node i of
 * request b) written to target_argmax [B][N], then dts_verify_tree_greedy
 * over it, in one call on `stream` (sources as for those two calls).
 *
 * Every other argument, output and error is as for dts_target_argmax and
 * dts_verify_tree_greedy; workspace is dts_target_argmax_workspace(B*N, vocab)
 * bytes.
 */
int dts_verify_tree_greedy_logits(const int32_t *draft_tokens, const float *logits, int vocab,
                                  int64_t row_stride, const int32_t *parents,
                                  const int32_t *next_token, const int32_t *next_sibling, int B,
                                  int N, int32_t *target_argmax, int32_t *accept_len,
                                  int32_t *accepted_path, int32_t *accepted_tokens,
                                  void *workspace, size_t ws_bytes, int32_t *err_dev,
                                  dts_stream_t stream);

/*
 * dts_sample_draws - the sampled target token of every verify row, drawn by
 * Gumbel-max keyed by position.
 *
 * Defined by [TS] "Sampled verify keys noise by position": a row's target
 * token is drawn by Gumbel-max keyed by (seed, position); for a tree the key
 * is the position the node predicts, vc + depth + 1, never its row, so the
 * token accepted at every position is the one plain decoding samples there.
 *
 *   logits       float [B*N][row_stride]  row b*N+i for node i of request b
 *   vc           int32 [B]     the pre-forward frontier (committed prefix length)
 *   depth        int32 [B][N]  node depths
 *   temperature  float [B]     T_b; T_b <= 0 or not finite: the plain argmax
 *   seed         uint64 [B]    the request's sampling seed
 *   draws        int32 [B][N]  out: argmax_v x_v * (1/T_b) + G(seed_b, vc_b + depth + 1, v)
 *   workspace    dts_target_argmax_workspace(B*N, vocab) bytes, as for
 *                dts_target_argmax
 *
 * G is fixed exactly, so that a draw is reproducible bit for bit: Philox4x32-10
 * (Salmon, Moraes, Dror and Shaw, SC 2011) with key (seed low word, seed high
 * word) and counter (v / 4, position, 0, 0), word v % 4 for vocabulary entry
 * v; u = (2 (word >> 9) + 1) 2^-24; G = -ln(-ln u), with ln and the scaling
 * evaluated in float32, one rounding per operation, by the series stated in
 * csrc/argmax.cu. Ties and NaN follow dts_target_argmax. Errors as for
 * dts_target_argmax; DTS_ERR_INVALID for a NULL vc, depth, temperature or seed.
 */
int dts_sample_draws(const float *logits, int vocab, int64_t row_stride, const int32_t *vc,
                     const int32_t *depth, const float *temperature, const uint64_t *seed, int B,
                     int N, int32_t *draws, void *workspace, size_t ws_bytes,
                     dts_stream_t stream);

/*
 * dts_verify_tree_sampled - dts_sample_draws, then dts_verify_tree_greedy over
 * the draws ([TS] "Sampled verify keys noise by position": acceptance is the
 * greedy tree walk over those draws, a child accepted when it equals its
 * parent's draw), in one call on `stream`. draws [B][N] is an output; every
 * other argument is as for those two calls.
 */
int dts_verify_tree_sampled(const int32_t *draft_tokens, const float *logits, int vocab,
                            int64_t row_stride, const int32_t *vc, const int32_t *depth,
                            const float *temperature, const uint64_t *seed,
                            const int32_t *parents, const int32_t *next_token,
                            const int32_t *next_sibling, int B, int N, int32_t *draws,
                            int32_t *accept_len, int32_t *accepted_path,
                            int32_t *accepted_tokens, void *workspace, size_t ws_bytes,
                            int32_t *err_dev, dts_stream_t stream);

/*
 * One K or V buffer of one layer (an entry of a cache group's address table).
 * Row s occupies bytes [base + s * slot_stride_bytes, ... + row_bytes).
 */
typedef struct dts_kv_buffer {
  void *base;                /* device address of slot 0 */
  int64_t slot_stride_bytes; /* bytes between consecutive slots */
  int64_t num_slots;         /* slots in this buffer (bounds check) */
  int32_t row_bytes;         /* bytes moved per slot; a multiple of 4 */
  int32_t reserved;          /* must be 0 */
} dts_kv_buffer;

/*
 * dts_compact_window_rows - move the accepted path's KV rows to the window's
 * leading slots in every buffer of the table.
 *
 * Defined by [TS] "The tree is a parameter of the chain path": the path's
 * target KV of every layer moves to the window's leading slots, by a word copy
 * that does not care about dtype, through a K/V address table per cache
 * group; [MI] "Discarding the rejected branches' KV": destinations are the
 * first accept_len window slots, sources the accepted nodes' slots.
 *
 *   table           dts_kv_buffer [n_buffers] in DEVICE memory
 *   write_locations int64 [B*N]   slot of window node i of request b
 *   accepted_path   int32 [B][N], accept_len int32 [B]  (dts_verify_tree_greedy)
 *
 * For t < accept_len[b]: row(write_locations[b*N+t]) <- row(write_locations[
 * b*N+path[t]]), read before anything is written (a path such as [0,2,3] reads
 * slot 2 for t=1 before writing it for t=2). Rows with path[t] == t do not
 * move. Each physical region moves once: an entry whose rows lie inside
 * another entry's rows (same stride; an aliased layer or a value view of a key
 * row) is skipped; entries that overlap only partly give DTS_DEV_BAD_BUFFER.
 * base and slot_stride_bytes must be multiples of 4 (16 gives the vector path).
 */
int dts_compact_window_rows(const dts_kv_buffer *table, int n_buffers,
                            const int64_t *write_locations, const int32_t *accepted_path,
                            const int32_t *accept_len, int B, int N, int32_t *err_dev,
                            dts_stream_t stream);

/*
 * dts_compact_rows - move the accepted path's hidden rows to the front of each
 * request's window and put the positions back to vc + i.
 *
 * Defined by [TS] "The tree is a parameter of the chain path" (hidden rows to
 * the front, positions from vc + depth back to vc + i) and "Position follows
 * depth" (the two position shifts cancel for any depth).
 *
 *   hidden     [B*N] rows of row_bytes bytes (row_bytes a multiple of 4)
 *   positions  int32 [B][N]   out: vc[b] + i for every i < N (may be NULL)
 *   vc         int32 [B]
 * For t < accept_len[b]: hidden[b*N+t] <- hidden[b*N+path[t]] (snapshot).
 */
int dts_compact_rows(void *hidden, int64_t row_bytes, int32_t *positions, const int32_t *vc,
                     const int32_t *accepted_path, const int32_t *accept_len, int B, int N,
                     int32_t *err_dev, dts_stream_t stream);

/*
 * dts_verify_prologue - dts_build_tree_mask and dts_write_window_kv (bf16
 * cache) in one launch, one warp per node. Each warp validates its request's
 * tree, forms its node's ancestor mask, position vc + depth, first child and
 * next sibling, and writes the node's rotated K and its V to the node's
 * window slot. The outputs, their layouts and the device-side errors are
 * exactly those of the two calls made in turn (with prefix_len for the slots
 * and vc for the positions, as there); arguments are validated as for those
 * calls.
 *
 *   parents, depth, vc            as for dts_build_tree_mask
 *   k_new, v_new, page_table, max_pages, page_size, prefix_len, Hkv, d,
 *   num_slots, rope_theta, k_cache, v_cache, write_locations
 *                                 as for dts_write_window_kv
 *   mask, positions, next_token, next_sibling   out, as for dts_build_tree_mask
 *
 * Sources as for the two calls ([TS] "One tree attention", "Position follows
 * depth, slot follows node index"; [AK] section one; [MI] "Building the mask,
 * for real", "Flattening, and the two link arrays").
 */
int dts_verify_prologue(const int32_t *parents, const int32_t *depth, const int32_t *vc,
                        const uint16_t *k_new, const uint16_t *v_new, const int32_t *page_table,
                        int max_pages, int page_size, const int32_t *prefix_len, int B, int N,
                        int Hkv, int d, int64_t num_slots, float rope_theta, uint64_t *mask,
                        int32_t *positions, int32_t *next_token, int32_t *next_sibling,
                        uint16_t *k_cache, uint16_t *v_cache, int64_t *write_locations,
                        int32_t *err_dev, dts_stream_t stream);

/*
 * dts_verify_epilogue - dts_verify_tree_greedy, dts_compact_window_rows and
 * dts_compact_rows in one launch: one block per (request, group of 8 KV
 * buffers); the block's first warp walks the request's tree, and the block
 * moves that request's KV rows (its group of the table) along the accepted
 * path; the first block of each request also moves the hidden rows and
 * resets the positions. The outputs and device-side errors are exactly those
 * of the three calls made in turn with the walk's outputs; arguments are
 * validated as for those calls.
 *
 *   draft_tokens, target_argmax, parents, next_token, next_sibling,
 *   accept_len, accepted_path, accepted_tokens
 *                                 as for dts_verify_tree_greedy
 *   table, n_buffers, write_locations   as for dts_compact_window_rows
 *                                 (n_buffers = 0: no KV rows move)
 *   hidden, row_bytes, positions, vc    as for dts_compact_rows
 *
 * Sources as for the three calls ([MI] "Walking the accepted path",
 * "Discarding the rejected branches' KV"; [AK] section two; [TS] "The tree is
 * a parameter of the chain path").
 */
int dts_verify_epilogue(const int32_t *draft_tokens, const int32_t *target_argmax,
                        const int32_t *parents, const int32_t *next_token,
                        const int32_t *next_sibling, int B, int N, int32_t *accept_len,
                        int32_t *accepted_path, int32_t *accepted_tokens,
                        const dts_kv_buffer *table, int n_buffers, const int64_t *write_locations,
                        void *hidden, int64_t row_bytes, int32_t *positions, const int32_t *vc,
                        int32_t *err_dev, dts_stream_t stream);

/*
 * dts_test_stall_attention - test hook, not a step of the verify path (the
 * pages have no counterpart). It lets a test make the tensor-core tree pass
 * give up on purpose, without a fault: with stall = 1, the pass's producer
 * issues no copy at all in the attention calls launched afterwards (every
 * tree/window attention entry point, bf16 and E4M3), so the waits of the other
 * roles run out after wait_budget_cycles; the kernel then frees its tensor
 * memory, returns, and *err_dev reads DTS_DEV_TIMEOUT. The outputs of such a
 * call are undefined. stall = 0 restores normal operation (the budget goes
 * back to about 2^31 cycles). The setting is process-wide; calls that overlap
 * with a change of it see either setting.
 *
 *   stall               0 or 1
 *   wait_budget_cycles  2^16 .. 2^31 (used only with stall = 1)
 *
 * Returns DTS_OK, or DTS_ERR_INVALID for values outside those ranges.
 */
int dts_test_stall_attention(int stall, long long wait_budget_cycles);

#ifdef __cplusplus
}
#endif

#endif /* DTS_H */
