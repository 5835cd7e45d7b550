/*
 * sgl_attn.h -- C ABI of the GB300 (sm_103a) slot-indexed attention library
 * (libsgl_attn.so).
 *
 * The library computes the data-parallel hot path of prefix-shared attention
 * over a token-granular KV pool: every token of every request owns one pool
 * slot, a table req_to_token[request row, position] gives that slot, and two
 * requests that share a prefix hold identical slot numbers in the leading
 * entries of their rows ("Inside SGLang", Step 3: Paged KV and the kernels
 * that read it; "Origins: the paper and the first commit", Memory: a
 * two-level pool paged by token).
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise.
 *     The caller allocates and owns all buffers; the library never allocates
 *     or frees device memory and never synchronises the device.
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream).
 *     The return value reports host-side argument validation and the launch
 *     status only; it never waits for the kernels.
 *   - bf16 tensors are dense, row-major, with the last dimension contiguous,
 *     and must start on a 16-byte boundary.  Indices are int32.
 *   - Index VALUES held in device memory (slots, req_to_token entries, lengths)
 *     are not read on the host.  Out-of-range values are undefined behaviour in
 *     the fast path; the sgl_check_* calls detect them without trapping.
 *   - head_dim must be 64 or 128; num_q_heads must be a multiple of
 *     num_kv_heads, with up to 128 query heads per KV head (decode runs a
 *     group of more than 16 as KV-head copies of at most 16 query heads
 *     each, every copy reading the KV head's rows).  Violations return SGL_ERR_UNSUPPORTED or
 *     SGL_ERR_INVALID_ARG before anything is launched.
 */
#ifndef SGL_ATTN_H
#define SGL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sgl_stream_t; /* == cudaStream_t */

typedef enum {
  SGL_OK = 0,
  SGL_ERR_INVALID_ARG = 1, /* null pointer, misaligned pointer, negative size */
  SGL_ERR_UNSUPPORTED = 2, /* head_dim / head-group shape not built */
  SGL_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  SGL_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
  SGL_ERR_INDEX = 5        /* reported by sgl_check_*: an index value is out of range */
} sgl_status;

typedef struct {
  int32_t num_q_heads;  /* Hq */
  int32_t num_kv_heads; /* Hkv; query head h reads KV head h / (Hq / Hkv) */
  int32_t head_dim;     /* D: 64 or 128 */
  int64_t pool_size;    /* S: number of slots in pool_k / pool_v */
  float sm_scale;       /* softmax scale; 0 selects 1/sqrt(head_dim) */
} sgl_attn_dims;

/* Human-readable name of a status code (static string, never NULL). */
const char* sgl_status_string(sgl_status status);

/* Library version, e.g. "0.1.0" (static string). */
const char* sgl_version(void);

/*
 * sgl_set_device_wait_limit_ns -- limit of the on-chip waits of the extend
 * and cascade-group kernels (failure detection; the pages have no
 * counterpart).
 *
 * Each stage barrier wait of sgl_extend_attention(_fp8) and of the group
 * pass of sgl_cascade_decode_attention(_fp8) gives up after this much wall
 * time (default 2 s): the kernel then records a nonzero code (0x5701) in the
 * status word of its workspace, lets its own copies and tensor-core work
 * finish, frees its tensor memory and returns, leaving that call's output
 * incomplete and the device usable.  A normal call's waits last
 * microseconds; a tiny limit makes them give up on purpose, which is how the
 * give-up path is tested.  ns == 0 restores the default.  Process-wide,
 * applies to launches made after the call (a captured CUDA graph keeps the
 * limit it was captured with); returns the previous limit.
 */
uint64_t sgl_set_device_wait_limit_ns(uint64_t ns);

/*
 * sgl_store_kv -- scatter new keys and values into their pool slots.
 *
 * Computes pool_k[slots[i], :, :] = k_new[i, :, :] and
 *          pool_v[slots[i], :, :] = v_new[i, :, :] for 0 <= i < n,
 * a bit-exact copy ("Origins: the paper and the first commit", Execution:
 * store_kv_cache writes the layer's K and V into the key and value buffers
 * at out_cache_loc).
 *   k_new, v_new : bf16 [n, Hkv, D]   new rows (read only)
 *   slots        : int32 [n]          distinct slots in [0, pool_size)
 *   pool_k/pool_v: bf16 [S, Hkv, D]   written at the n slots only
 * Duplicate slots are a precondition violation (the last writer is not
 * defined).  n == 0 is a no-op.
 */
sgl_status sgl_store_kv(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                        void* pool_k, void* pool_v, const sgl_attn_dims* dims,
                        sgl_stream_t stream);

/*
 * sgl_extend_attention -- attention of new suffix tokens over a cached prefix.
 *
 * For request r (0 <= r < batch) with prefix length p = prefix_lens[r],
 * extend length e = extend_lens[r] and row = req_pool_idx[r]:
 *   keys/values 0..p-1  : pool_k/pool_v[req_to_token[row * rtt_stride + j]]
 *   keys/values p..p+e-1: k_new/v_new rows of the request's suffix
 * Suffix query i (0 <= i < e; absolute position p+i) attends to keys
 * 0..p+i, so the result equals the last e rows of full causal attention over
 * the p+e tokens ("Inside SGLang", Step 3: Look inside the forward pass --
 * scores scaled by 1/sqrt(head_dim), keys after the query masked, softmax,
 * times V; "Origins", Batching: EXTEND computes only the new suffix after the
 * cached prefix, seq_len = prefix + extend).
 *   q            : bf16 [T, Hq, D]    suffix queries of all requests back to
 *                                    back (request r starts at the exclusive
 *                                    prefix sum of extend_lens)
 *   k_new, v_new : bf16 [T, Hkv, D]   suffix keys/values, same order
 *   pool_k/pool_v: bf16 [S, Hkv, D]   read at prefix slots only (never written)
 *   req_to_token : int32 [rtt_rows, rtt_stride]
 *   req_pool_idx, prefix_lens, extend_lens: int32 [batch]
 *   total_extend : T = sum(extend_lens)  (host value; sizes the launch)
 *   max_extend   : >= max(extend_lens)   (host value)
 *   max_prefix   : >= max(prefix_lens)   (host value; informational)
 *   out          : bf16 [T, Hq, D]    written for every suffix row
 *   workspace    : device buffer of at least sgl_extend_workspace_bytes();
 *                  it must be zero-filled once before first use.  Word 0 is
 *                  set to a nonzero code if a bounded on-chip wait gave up
 *                  (the output is then incomplete); it is never cleared by
 *                  the library.
 * Softmax is computed in fp32 from fp32 tensor-core accumulators; out is
 * rounded to bf16 (nearest even).
 */
sgl_status sgl_extend_attention(const void* q, const void* k_new, const void* v_new,
                                const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                                int32_t max_extend, int32_t max_prefix, void* out, void* workspace,
                                size_t workspace_bytes, const sgl_attn_dims* dims,
                                sgl_stream_t stream);

/*
 * sgl_decode_attention -- one query per request over all of its slots.
 *
 * out[r, h] = softmax_j(scale * q[r, h] . K_j) . V_j over j < seq_lens[r],
 * K_j/V_j = pool rows at req_to_token[req_pool_idx[r] * rtt_stride + j]
 * ("Inside SGLang", Step 3: decode reads the key and value of every earlier
 * token).  seq_lens[r] counts the new token, whose K/V sgl_store_kv must
 * have written first (decode equals extend with extend_len = 1).
 *   q            : bf16 [batch, Hq, D]
 *   seq_lens     : int32 [batch], each >= 1
 *   max_seq_len  : >= max(seq_lens) (host value; sizes the split-KV schedule)
 *   out          : bf16 [batch, Hq, D]
 *   workspace    : >= sgl_decode_workspace_bytes(batch, max_seq_len, dims);
 *                  scratch for the split-KV partial results.
 * The keys of a request are split into chunks processed in parallel; each
 * chunk keeps an fp32 online-softmax state (max, sum, weighted V sum) and a
 * second kernel merges the chunks of requests that have more than one.
 */
sgl_status sgl_decode_attention(const void* q, const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* seq_lens,
                                int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                                size_t workspace_bytes, const sgl_attn_dims* dims,
                                sgl_stream_t stream);

/*
 * sgl_decode_attention_noalloc -- sgl_decode_attention for callers that
 * cannot allocate device memory.  The paper has no counterpart: this is a
 * deployment variant of the decode entry point above.
 *
 * Some callers may not call cudaMalloc (or any allocating routine) while they
 * run attention -- runtimes whose memory planner fixes every device buffer at
 * start-up, and plugin-style hosts that pass a kernel only its inputs and
 * outputs -- so they cannot provide the decode workspace.  This call computes
 * exactly what sgl_decode_attention computes, with the same arguments minus
 * the workspace, and takes its split-KV scratch from a fixed array of
 * SGL_DECODE_NOALLOC_SCRATCH_BYTES in the library's own device memory.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - Every GPU that loads the library's module holds the array until the
 *     process exits.
 *   - Arguments are checked exactly as sgl_decode_attention checks them,
 *     with the same error codes (a shape the kernels are not built for is
 *     SGL_ERR_UNSUPPORTED).  Then work whose scratch need
 *     (sgl_decode_workspace_bytes(batch, max_seq_len, dims)) exceeds
 *     SGL_DECODE_NOALLOC_SCRATCH_BYTES is rejected with SGL_ERR_WORKSPACE
 *     before anything is launched; use sgl_decode_attention with a caller
 *     workspace for it.
 *   - The first call on a device, in each CUDA context, looks up the array's
 *     device address there (the device must be current); make that first
 *     call before any stream capture.  A device reset (cudaDeviceReset)
 *     after the first call is not supported: the library's module is loaded
 *     again at an address the cached lookup does not know.
 *   - All calls share the array and it keeps the last call's contents:
 *     calls whose kernels overlap on the GPU race and must be serialised by
 *     the caller (one stream, or explicit ordering).  No part of it needs
 *     clearing between calls.
 */
#define SGL_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
sgl_status sgl_decode_attention_noalloc(const void* q, const void* pool_k, const void* pool_v,
                                        const int32_t* req_to_token, int32_t rtt_rows,
                                        int32_t rtt_stride, const int32_t* req_pool_idx,
                                        const int32_t* seq_lens, int32_t batch,
                                        int32_t max_seq_len, void* out, const sgl_attn_dims* dims,
                                        sgl_stream_t stream);

/*
 * sgl_mixed_attention -- the extend batch and the decode batch of one step in
 * one launch ("Inside SGLang", Step 10: Split long prompts into chunks: a
 * prefill chunk and the running requests' decode tokens share a forward pass;
 * "A walkthrough of SGLang": the MIXED forward mode).
 *
 * Computes exactly what sgl_extend_attention (the q_ext .. out_ext arguments,
 * ext_workspace as its workspace) and sgl_decode_attention (q_dec .. out_dec,
 * dec_workspace) compute over the same bf16 pools and req_to_token -- the same
 * kernels' arithmetic on the same tiles and work items, so the outputs are
 * those two calls' outputs bit for bit.  The extend is bound by the tensor
 * cores and the decode by HBM bandwidth; here they share the GPU's SMs in one
 * persistent launch: extend_sms SMs start on extend tiles, the others on
 * decode work, and an SM whose side has run out takes the other side's work.
 * extend_sms = 0 picks the split from the host values (half the maxima taken
 * as mean lengths); a positive extend_sms sets it (from the SM count on, every
 * SM starts on extend tiles).  Measured: the launch takes the same time at
 * every split (the SMs' work adds up whichever side they start on).
 *   - The pools are bf16; the argument checks, preconditions, error codes and
 *     workspace sizes are those of the two calls (ext_workspace >=
 *     sgl_extend_workspace_bytes, its first 256 bytes zero-filled once before
 *     first use: word 0 is the extend's bounded-wait status, words 1..3 the
 *     launch's work counters, reset by the launch itself).
 *   - Either batch may be empty (the other call alone runs).  Decode groups of
 *     1 or 2 query heads per KV head at head_dim 64 or 128 run in the single
 *     launch; other shapes run the two calls' kernels one after the other.
 *   - The store of the step's new K/V (sgl_store_kv) must precede the call, as
 *     for a decode.
 */
sgl_status sgl_mixed_attention(
    const void* q_ext, const void* k_new, const void* v_new, const int32_t* ext_req_pool_idx,
    const int32_t* prefix_lens, const int32_t* extend_lens, int32_t ext_batch, int32_t total_extend,
    int32_t max_extend, int32_t max_prefix, void* out_ext, void* ext_workspace, size_t ext_workspace_bytes,
    const void* q_dec, const int32_t* dec_req_pool_idx, const int32_t* seq_lens, int32_t dec_batch,
    int32_t max_seq_len, void* out_dec, void* dec_workspace, size_t dec_workspace_bytes, const void* pool_k,
    const void* pool_v, const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride, int32_t extend_sms,
    const sgl_attn_dims* dims, sgl_stream_t stream);

/*
 * sgl_cascade_decode_attention -- decode attention that reads each shared
 * prefix once per group of requests.
 *
 * Computes what sgl_decode_attention computes (same arguments, same output),
 * given a description of the keys that several requests of the batch share.
 * Requests that share a prefix hold identical slot numbers in the leading
 * entries of their rows ("Inside SGLang", Step 3: Paged KV and the kernels
 * that read it), so the softmax over a request's keys splits into one state
 * per shared group plus one for its private tail, merged exactly (the
 * regrouping of the softmax sums that also joins the split-KV chunks).  A
 * group's keys are gathered once and all of its members' query heads attend
 * to them on the tensor cores; the tails run as plain split-KV decode.
 *   group_start, group_len : int32 [n_groups]  group j covers positions
 *                            [group_start[j], group_start[j] + group_len[j])
 *                            of every member's row; group_len >= 1
 *   group_depth            : int32 [n_groups]  j's rank among each member's
 *                            groups, in [0, max_depth)
 *   group_member_off       : int32 [n_groups + 1]  CSR offsets (first 0)
 *   group_members          : int32 [group_member_off[n_groups]]  member
 *                            requests (indices into the batch)
 *   n_groups               : host value (<= 65535); 0 = plain decode
 *   max_group_members      : >= the largest member count (host; sizes the grid)
 *   max_depth              : >= the largest group_depth + 1 (host; sizes the
 *                            workspace)
 *   workspace              : >= sgl_cascade_decode_workspace_bytes(batch,
 *                            max_seq_len, max_depth, dims); the first 256
 *                            bytes must be zero-filled once before first use:
 *                            word 0 is set to a nonzero code if a bounded
 *                            on-chip wait of the group pass gave up (the
 *                            output is then incomplete); it is never cleared.
 * Preconditions (sgl_check_cascade_groups verifies them): every member's row
 * holds the same slots as the group's first member over the group's range
 * (the keys are read from the first member's row); each request's groups,
 * ordered by depth 0, 1, ..., cover [0, shared_len) back to back with
 * shared_len <= seq_len; a request's keys [shared_len, seq_len) are its
 * private tail (possibly empty).  A request in no group is plain decode.
 * Member indices outside [0, batch) and depths outside [0, max_depth) are
 * skipped; other violations give undefined results but no out-of-bounds
 * write.
 */
sgl_status sgl_cascade_decode_attention(
    const void* q, const void* pool_k, const void* pool_v, const int32_t* req_to_token,
    int32_t rtt_rows, int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
    int32_t batch, int32_t max_seq_len, const int32_t* group_start, const int32_t* group_len,
    const int32_t* group_depth, const int32_t* group_member_off, const int32_t* group_members,
    int32_t n_groups, int32_t max_group_members, int32_t max_depth, void* out, void* workspace,
    size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream);

/*
 * FP8 KV pool ("Inside SGLang", Step 6: Decide how much memory becomes KV
 * cache -- with --kv-cache-dtype fp8_e4m3 each token's K and V take half the
 * bytes; the attention kernels read FP8 directly, and K and V carry one scale
 * each, from the checkpoint, 1.0 when missing).
 *
 * Pool rows hold e4m3 codes (uint8 [S, Hkv, D]: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals, no infinities, largest finite 448); a
 * code c of pool_k stands for the value e4m3(c) * k_scale (pool_v: v_scale).
 *
 * sgl_store_kv_fp8 -- pool_k[slots[i]] = e4m3(k_new[i] / k_scale), likewise
 *   V: the quotient in IEEE float32, rounded to e4m3 to nearest (ties to
 *   even), saturating to +-448.  k_new, v_new bf16 [n, Hkv, D]; slots as in
 *   sgl_store_kv; scales finite and > 0 (else SGL_ERR_INVALID_ARG).
 * sgl_decode_attention_fp8 -- sgl_decode_attention over an e4m3 pool: the
 *   keys and values are code * scale; q, out and the workspace as there
 *   (sgl_decode_workspace_bytes).  The K scale is folded into the query and
 *   the V scale into the output; accumulation is fp32.
 * sgl_extend_attention_fp8 -- sgl_extend_attention over an e4m3 pool.  Every
 *   key and value is read from the pool through req_to_token: request r's
 *   row holds its prefix slots at positions 0..p-1 AND its suffix slots at
 *   positions p..p+e-1, already written by sgl_store_kv_fp8 (so an extend,
 *   a later decode and a cascade decode all see the same stored values of a
 *   position; there is no k_new / v_new argument).  Suffix query i attends to
 *   positions 0..p+i.  q, out, lengths, workspace as for sgl_extend_attention.
 *   The codes are widened exactly to f16 tensor-core operands; the query is
 *   widened from bf16 to f16 (exact for |q| in [2^-14, 65504]; smaller values
 *   round as f16 subnormals, |q| > 65504 is outside the supported range) and
 *   P is rounded to f16; accumulation is fp32.  Index check:
 *   sgl_check_extend_fp8_indices (it covers the suffix positions too).
 * sgl_cascade_decode_attention_fp8 -- sgl_cascade_decode_attention over an
 *   e4m3 pool (group pass on f16 tensor-core operands as above, tails and
 *   combine as sgl_decode_attention_fp8); same arguments, groups, workspace
 *   (sgl_cascade_decode_workspace_bytes) and preconditions.
 */
sgl_status sgl_store_kv_fp8(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                            void* pool_k, void* pool_v, float k_scale, float v_scale,
                            const sgl_attn_dims* dims, sgl_stream_t stream);
sgl_status sgl_decode_attention_fp8(const void* q, const void* pool_k, const void* pool_v,
                                    float k_scale, float v_scale, const int32_t* req_to_token,
                                    int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                                    size_t workspace_bytes, const sgl_attn_dims* dims,
                                    sgl_stream_t stream);
sgl_status sgl_extend_attention_fp8(const void* q, const void* pool_k, const void* pool_v,
                                    float k_scale, float v_scale, const int32_t* req_to_token,
                                    int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                    const int32_t* extend_lens, int32_t batch,
                                    int32_t total_extend, int32_t max_extend, int32_t max_prefix,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    const sgl_attn_dims* dims, sgl_stream_t stream);
sgl_status sgl_cascade_decode_attention_fp8(
    const void* q, const void* pool_k, const void* pool_v, float k_scale, float v_scale,
    const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
    const int32_t* req_pool_idx, const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
    const int32_t* group_start, const int32_t* group_len, const int32_t* group_depth,
    const int32_t* group_member_off, const int32_t* group_members, int32_t n_groups,
    int32_t max_group_members, int32_t max_depth, void* out, void* workspace,
    size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream);

/* Workspace sizes (host only; no device call). */
size_t sgl_extend_workspace_bytes(int32_t batch, int32_t total_extend, const sgl_attn_dims* dims);
size_t sgl_decode_workspace_bytes(int32_t batch, int32_t max_seq_len, const sgl_attn_dims* dims);
size_t sgl_cascade_decode_workspace_bytes(int32_t batch, int32_t max_seq_len, int32_t max_depth,
                                          const sgl_attn_dims* dims);

/*
 * Checked mode.  Each call validates the index values in device memory with a
 * kernel that never traps: it writes into d_error (int32[4], device) the
 * first violation found as {kind, a, b, c} and leaves d_error untouched when
 * everything is in range.  The caller zeroes d_error beforehand and reads it
 * after the stream completes; kind != 0 means SGL_ERR_INDEX.
 *   kind 1: slot out of [0, pool_size)          a = list/row index, b = position, c = value
 *   kind 2: req_pool_idx out of [0, rtt_rows)   a = request, c = value
 *   kind 3: length negative / seq_len < 1        a = request, c = value
 *   kind 4: prefix+extend or seq_len > rtt_stride  a = request, c = length
 *   kind 5: sum(extend_lens) != total_extend or a length above the host max
 *   kind 6: duplicate slot in one store_kv call  a = second index, c = slot
 *   kind 7: malformed cascade group (offsets, member count above the host
 *           max, member outside the batch, depth outside [0, max_depth),
 *           length < 1)                      a = group, b = which check, c = value
 *   kind 8: group range past a member's seq_len or past rtt_stride
 *                                            a = group, b = member (-1: stride), c = end
 *   kind 9: a member's slot differs from the first member's (not shared)
 *                                            a = group, b = position, c = member
 *   kind 10: a request's groups do not cover [0, shared_len) back to back
 *           (two groups at one depth, a gap, or a wrong start)
 *                                            a = request, b = depth, c = group / start
 * sgl_check_extend_indices checks the slots of positions 0..p-1 of each row
 * (the ones sgl_extend_attention reads); sgl_check_extend_fp8_indices those
 * of positions 0..p+e-1 (sgl_extend_attention_fp8 reads the suffix from the
 * pool too).
 * sgl_check_store_kv_indices needs a scratch bitmap of (pool_size+7)/8 bytes
 * (rounded up to 16) in `bitmap`; it is cleared by the call.
 * sgl_check_cascade_groups needs sgl_check_cascade_scratch_bytes(batch,
 * max_depth) bytes of scratch (overwritten by the call); it checks the
 * groups only -- pair it with sgl_check_decode_indices for rows, lengths and
 * slot ranges.
 */
sgl_status sgl_check_store_kv_indices(const int32_t* slots, int32_t n, int64_t pool_size,
                                      void* bitmap, size_t bitmap_bytes, int32_t* d_error,
                                      sgl_stream_t stream);
sgl_status sgl_check_extend_indices(const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                    const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                                    int32_t max_extend, int32_t max_prefix, int64_t pool_size,
                                    int32_t* d_error, sgl_stream_t stream);
sgl_status sgl_check_extend_fp8_indices(const int32_t* req_to_token, int32_t rtt_rows,
                                        int32_t rtt_stride, const int32_t* req_pool_idx,
                                        const int32_t* prefix_lens, const int32_t* extend_lens,
                                        int32_t batch, int32_t total_extend, int32_t max_extend,
                                        int32_t max_prefix, int64_t pool_size, int32_t* d_error,
                                        sgl_stream_t stream);
sgl_status sgl_check_decode_indices(const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, int64_t pool_size,
                                    int32_t* d_error, sgl_stream_t stream);
size_t sgl_check_cascade_scratch_bytes(int32_t batch, int32_t max_depth);
sgl_status sgl_check_cascade_groups(const int32_t* req_to_token, int32_t rtt_rows,
                                    int32_t rtt_stride, const int32_t* req_pool_idx,
                                    const int32_t* seq_lens, int32_t batch,
                                    const int32_t* group_start, const int32_t* group_len,
                                    const int32_t* group_depth, const int32_t* group_member_off,
                                    const int32_t* group_members, int32_t n_groups,
                                    int32_t max_group_members, int32_t max_depth, void* scratch,
                                    size_t scratch_bytes, int32_t* d_error, sgl_stream_t stream);

/*
 * Radix tree of cached token runs (host only; no device memory, no CUDA call).
 *
 * The structure that lays out req_to_token rows ("Inside SGLang", Step 4:
 * Grow a prefix tree, then run out of room; "SGLang" notes, RadixAttention
 * and Eviction): each node holds a run of token ids, the KV-pool slots of
 * those tokens, children keyed by first token, and a lock count.
 *   match_prefix -- walk down while tokens agree; if the match ends inside a
 *                   node, split it there.  Returns the matched length m
 *                   (-1 on a bad argument), writes the path's slots
 *                   (min(m, cap) of them) and the last matched node's handle
 *                   (the root when m = 0).  Every node passed gets a new
 *                   access time.
 *   insert       -- the same walk, then the unmatched rest becomes a leaf
 *                   holding slots[m..n).  Returns m: slots[0..m) duplicate
 *                   cached tokens and are the caller's to free.
 *   inc/dec_lock_ref -- lock (unlock) a node and its path to the root; a
 *                   running request locks the last node it matched.  A split
 *                   copies the lock count to the new prefix node.  Stale
 *                   handles (of evicted nodes) and unbalanced decrements
 *                   return SGL_ERR_INVALID_ARG and change nothing.
 *   evict        -- free unlocked leaves, least recently used first (access
 *                   times from a logical clock; ties by creation order), a
 *                   parent that becomes a leaf joining the candidates, until
 *                   at least num_tokens tokens are freed, nothing evictable is
 *                   left, or the next leaf would not fit in `cap`.  Writes the
 *                   freed slots (each leaf's in token order) and returns their
 *                   count.
 *   groups       -- the shared-prefix groups of a decode batch whose request
 *                   r matched node nodes[r]: every non-root node on two or
 *                   more requests' paths (start = position of its first token,
 *                   len = its run, depth = its rank on the paths, members in
 *                   ascending order), listed by (depth, start, first member) --
 *                   the input of sgl_cascade_decode_attention.  Returns the
 *                   group count and sets *n_members_out; the arrays
 *                   (member_off holds n_groups + 1 entries) are written only
 *                   when the counts fit cap_groups and cap_members.
 * A tree is not thread-safe: one thread (the scheduler) owns it.
 */
typedef struct sgl_radix_tree sgl_radix_tree;
sgl_radix_tree* sgl_radix_create(void);
void sgl_radix_destroy(sgl_radix_tree* tree);
int32_t sgl_radix_match_prefix(sgl_radix_tree* tree, const int32_t* tokens, int32_t n,
                               int32_t* slots_out, int32_t cap, int64_t* node_out);
int32_t sgl_radix_insert(sgl_radix_tree* tree, const int32_t* tokens, const int32_t* slots,
                         int32_t n);
sgl_status sgl_radix_inc_lock_ref(sgl_radix_tree* tree, int64_t node);
sgl_status sgl_radix_dec_lock_ref(sgl_radix_tree* tree, int64_t node);
int32_t sgl_radix_evict(sgl_radix_tree* tree, int32_t num_tokens, int32_t* slots_out, int32_t cap);
int64_t sgl_radix_evictable_tokens(const sgl_radix_tree* tree);
int64_t sgl_radix_protected_tokens(const sgl_radix_tree* tree);
int32_t sgl_radix_groups(const sgl_radix_tree* tree, const int64_t* nodes, int32_t batch,
                         int32_t* group_start, int32_t* group_len, int32_t* group_depth,
                         int32_t* member_off, int32_t* members, int32_t cap_groups,
                         int32_t cap_members, int32_t* n_members_out);

#ifdef __cplusplus
}
#endif

#endif /* SGL_ATTN_H */
