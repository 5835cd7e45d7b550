// C ABI of libsgl_attn.so: host-side argument validation, workspace sizing,
// dispatch to the kernel launchers, and the checked-mode index validators.
// Nothing here allocates device memory or synchronises the device.
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace sgl {

namespace {
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

uint64_t device_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_kv_scale(float s) { return s > 0.f && !isinf(s) && !isnan(s); }

// Validates dims and fills the effective scale; returns SGL_OK or an error.
sgl_status check_dims(const sgl_attn_dims* d, float* scale) {
  if (d == nullptr) return SGL_ERR_INVALID_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->pool_size <= 0) return SGL_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return SGL_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return SGL_ERR_UNSUPPORTED;
  if (!(d->sm_scale >= 0.f) || isinf(d->sm_scale)) return SGL_ERR_INVALID_ARG;
  *scale = d->sm_scale > 0.f ? d->sm_scale : 1.0f / sqrtf((float)d->head_dim);
  return SGL_OK;
}

__device__ void report(int32_t* err, int32_t kind, int32_t a, int32_t b, int32_t c) {
  if (atomicCAS(err, 0, kind) == 0) {
    err[1] = a;
    err[2] = b;
    err[3] = c;
  }
}

__global__ void check_store_kernel(const int32_t* __restrict__ slots, int32_t n, int64_t S,
                                   uint32_t* __restrict__ bitmap, int32_t* err) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = slots[i];
    if (s < 0 || s >= S) {
      report(err, 1, (int32_t)i, 0, s);
      continue;
    }
    const uint32_t bit = 1u << (s & 31);
    const uint32_t old = atomicOr(&bitmap[s >> 5], bit);
    if (old & bit) report(err, 6, (int32_t)i, 0, s);
  }
}

// mode 0: extend (lens_a = prefix, lens_b = extend; the prefix slots are read);
// mode 2: the same over an e4m3 pool (prefix and suffix slots are read);
// mode 1: decode (lens_a = seq)
__global__ void check_rows_kernel(const int32_t* __restrict__ rtt, int32_t rtt_rows, int32_t stride,
                                  const int32_t* __restrict__ rpi, const int32_t* __restrict__ lens_a,
                                  const int32_t* __restrict__ lens_b, int32_t mode, int64_t S,
                                  int32_t max_a, int32_t max_b, int32_t* err) {
  const int r = blockIdx.x;
  const int32_t row = rpi[r];
  if (row < 0 || row >= rtt_rows) {
    if (threadIdx.x == 0) report(err, 2, r, 0, row);
    return;
  }
  int32_t n;
  if (mode != 1) {
    const int32_t pl = lens_a[r], el = lens_b[r];
    if (pl < 0 || el < 0) {
      if (threadIdx.x == 0) report(err, 3, r, 0, pl < 0 ? pl : el);
      return;
    }
    if ((int64_t)pl + el > stride) {
      if (threadIdx.x == 0) report(err, 4, r, 0, pl + el);
      return;
    }
    if (pl > max_a || el > max_b) {
      if (threadIdx.x == 0) report(err, 5, r, 0, pl > max_a ? pl : el);
      return;
    }
    n = mode == 2 ? pl + el : pl;
  } else {
    const int32_t sl = lens_a[r];
    if (sl < 1) {
      if (threadIdx.x == 0) report(err, 3, r, 0, sl);
      return;
    }
    if (sl > stride) {
      if (threadIdx.x == 0) report(err, 4, r, 0, sl);
      return;
    }
    if (sl > max_a) {
      if (threadIdx.x == 0) report(err, 5, r, 0, sl);
      return;
    }
    n = sl;
  }
  const int32_t* row_p = rtt + (int64_t)row * stride;
  for (int32_t j = threadIdx.x; j < n; j += blockDim.x) {
    const int32_t s = row_p[j];
    if (s < 0 || s >= S) report(err, 1, r, j, s);
  }
}

__global__ void check_sum_kernel(const int32_t* __restrict__ lens, int32_t batch, int32_t total,
                                 int32_t* err) {
  __shared__ long long part[32];
  long long s = 0;
  for (int i = threadIdx.x; i < batch; i += blockDim.x) s += lens[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long t = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
    if (t != total) report(err, 5, -1, (int32_t)t, total);
  }
}

// Cascade groups, one block per group (grid-stride): structure, member
// ranges, shared slots, and each (request, depth) claimed by one group only.
__global__ void check_groups_kernel(const int32_t* __restrict__ rtt, int32_t rtt_rows,
                                    int32_t stride, const int32_t* __restrict__ rpi,
                                    const int32_t* __restrict__ seq_lens, int32_t batch,
                                    const int32_t* __restrict__ gstart,
                                    const int32_t* __restrict__ glen,
                                    const int32_t* __restrict__ gdepth,
                                    const int32_t* __restrict__ moff,
                                    const int32_t* __restrict__ mem, int32_t n_groups,
                                    int32_t max_members, int32_t max_depth,
                                    int32_t* __restrict__ owner, int32_t* err) {
  __shared__ int bad;
  if (blockIdx.x == 0 && threadIdx.x == 0 && moff[0] != 0) report(err, 7, 0, 0, moff[0]);
  for (int32_t j = blockIdx.x; j < n_groups; j += gridDim.x) {
    const int32_t a = moff[j], b = moff[j + 1];
    const int32_t st = gstart[j], ln = glen[j], dp = gdepth[j];
    if (threadIdx.x == 0) {
      bad = 0;
      if (b < a || b - a > max_members) bad = 1, report(err, 7, j, 0, b - a);
      else if (dp < 0 || dp >= max_depth) bad = 1, report(err, 7, j, 1, dp);
      else if (ln < 1 || st < 0) bad = 1, report(err, 7, j, 2, ln < 1 ? ln : st);
      else if ((int64_t)st + ln > stride) bad = 1, report(err, 8, j, -1, st + ln);
    }
    __syncthreads();
    if (!bad) {
      for (int32_t k = a + threadIdx.x; k < b; k += blockDim.x) {
        const int32_t r = mem[k];
        if (r < 0 || r >= batch) {
          report(err, 7, j, 3, r);
          atomicOr(&bad, 1);
          continue;
        }
        const int32_t row = rpi[r];
        if (row < 0 || row >= rtt_rows) {
          report(err, 2, r, 0, row);
          atomicOr(&bad, 1);
          continue;
        }
        if (st + ln > seq_lens[r]) report(err, 8, j, r, st + ln);
        if (atomicCAS(&owner[(int64_t)r * max_depth + dp], -1, j) != -1) report(err, 10, r, dp, j);
      }
    }
    __syncthreads();
    if (!bad && b > a) {
      const int32_t* ref = rtt + (int64_t)rpi[mem[a]] * stride + st;
      const int64_t n = (int64_t)(b - a - 1) * ln;
      for (int64_t t = threadIdx.x; t < n; t += blockDim.x) {
        const int32_t r = mem[a + 1 + (int32_t)(t / ln)];
        const int32_t i = (int32_t)(t % ln);
        if (rtt[(int64_t)rpi[r] * stride + st + i] != ref[i]) report(err, 9, j, st + i, r);
      }
    }
    __syncthreads();
  }
}

// Each request's groups, by depth, must cover [0, shared_len) back to back.
__global__ void check_tiling_kernel(const int32_t* __restrict__ owner, int32_t batch,
                                    int32_t max_depth, const int32_t* __restrict__ gstart,
                                    const int32_t* __restrict__ glen, int32_t* err) {
  const int32_t r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= batch) return;
  int32_t pos = 0;
  bool ended = false;
  for (int32_t d = 0; d < max_depth; ++d) {
    const int32_t j = owner[(int64_t)r * max_depth + d];
    if (j < 0) {
      ended = true;
      continue;
    }
    if (ended || gstart[j] != pos) {
      report(err, 10, r, d, gstart[j]);
      return;
    }
    pos += glen[j];
  }
}

sgl_status last_launch() { return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA; }

}  // namespace

// Every host-side check of a decode call except the workspace's: dims, the
// head-group shape the kernels are built for, sizes, pointers and alignment.
// SGL_OK with batch == 0 means there is nothing to launch.
sgl_status validate_decode_call(const void* q, const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* seq_lens, int32_t batch,
                                int32_t max_seq_len, const void* out, const sgl_attn_dims* dims,
                                float* scale) {
  sgl_status st = check_dims(dims, scale);
  if (st != SGL_OK) return st;
  if (batch < 0 || max_seq_len < 0) return SGL_ERR_INVALID_ARG;
  if (batch == 0) return SGL_OK;
  if (max_seq_len < 1) return SGL_ERR_INVALID_ARG;
  if (!q || !pool_k || !pool_v || !req_to_token || !req_pool_idx || !seq_lens || !out)
    return SGL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool_k) || !aligned16(pool_v)) return SGL_ERR_INVALID_ARG;
  if (rtt_rows <= 0 || rtt_stride <= 0) return SGL_ERR_INVALID_ARG;
  return decode_shape_supported(dims->num_q_heads, dims->num_kv_heads);
}
}  // namespace sgl

using namespace sgl;

extern "C" {

const char* sgl_status_string(sgl_status s) {
  switch (s) {
    case SGL_OK: return "SGL_OK";
    case SGL_ERR_INVALID_ARG: return "SGL_ERR_INVALID_ARG";
    case SGL_ERR_UNSUPPORTED: return "SGL_ERR_UNSUPPORTED";
    case SGL_ERR_WORKSPACE: return "SGL_ERR_WORKSPACE";
    case SGL_ERR_CUDA: return "SGL_ERR_CUDA";
    case SGL_ERR_INDEX: return "SGL_ERR_INDEX";
  }
  return "SGL_ERR_UNKNOWN";
}

const char* sgl_version(void) { return "0.1.0"; }

uint64_t sgl_set_device_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

sgl_status sgl_store_kv(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                        void* pool_k, void* pool_v, const sgl_attn_dims* dims,
                        sgl_stream_t stream) {
  float scale;
  sgl_status st = check_dims(dims, &scale);
  if (st != SGL_OK) return st;
  if (n < 0) return SGL_ERR_INVALID_ARG;
  if (n == 0) return SGL_OK;
  if (!k_new || !v_new || !slots || !pool_k || !pool_v) return SGL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool_k) || !aligned16(pool_v))
    return SGL_ERR_INVALID_ARG;
  if ((int64_t)n > dims->pool_size) return SGL_ERR_INVALID_ARG;  // slots must be distinct
  const int32_t row_bytes = dims->num_kv_heads * dims->head_dim * 2;
  return launch_store_kv(k_new, v_new, slots, n, pool_k, pool_v, row_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

sgl_status sgl_store_kv_fp8(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                            void* pool_k, void* pool_v, float k_scale, float v_scale,
                            const sgl_attn_dims* dims, sgl_stream_t stream) {
  float scale;
  sgl_status st = check_dims(dims, &scale);
  if (st != SGL_OK) return st;
  if (n < 0 || !valid_kv_scale(k_scale) || !valid_kv_scale(v_scale)) return SGL_ERR_INVALID_ARG;
  if (n == 0) return SGL_OK;
  if (!k_new || !v_new || !slots || !pool_k || !pool_v) return SGL_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool_k) || !aligned16(pool_v))
    return SGL_ERR_INVALID_ARG;
  if ((int64_t)n > dims->pool_size) return SGL_ERR_INVALID_ARG;
  return launch_store_kv_fp8(k_new, v_new, slots, n, pool_k, pool_v,
                             dims->num_kv_heads * dims->head_dim, k_scale, v_scale,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t sgl_extend_workspace_bytes(int32_t batch, int32_t total_extend, const sgl_attn_dims* dims) {
  (void)batch;
  (void)total_extend;
  (void)dims;
  return extend_workspace_bytes();
}

size_t sgl_decode_workspace_bytes(int32_t batch, int32_t max_seq_len, const sgl_attn_dims* dims) {
  if (dims == nullptr || dims->num_kv_heads <= 0 || dims->num_q_heads <= 0) return 0;
  return decode_workspace_bytes(batch, max_seq_len, dims->num_q_heads, dims->num_kv_heads,
                                dims->head_dim);
}

size_t sgl_cascade_decode_workspace_bytes(int32_t batch, int32_t max_seq_len, int32_t max_depth,
                                          const sgl_attn_dims* dims) {
  if (dims == nullptr || dims->num_kv_heads <= 0 || dims->num_q_heads <= 0 || max_depth < 0)
    return 0;
  return decode_workspace_bytes(batch, max_seq_len, dims->num_q_heads, dims->num_kv_heads,
                                dims->head_dim, true, max_depth);
}

namespace {
// k_new / v_new are null on an e4m3 pool (the suffix is read from the pool)
// Host checks of an extend call; fills *a.  *empty: nothing to launch.
sgl_status extend_args(const void* q, const void* k_new, const void* v_new, const void* pool_k,
                       const void* pool_v, bool kv_fp8, float k_scale, float v_scale,
                       const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                       const int32_t* req_pool_idx, const int32_t* prefix_lens,
                       const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                       int32_t max_extend, int32_t max_prefix, void* out, void* workspace,
                       size_t workspace_bytes, const sgl_attn_dims* dims, ExtendArgs* ap, bool* empty) {
  float scale;
  sgl_status st = check_dims(dims, &scale);
  if (st != SGL_OK) return st;
  if (batch < 0 || total_extend < 0 || max_extend < 0 || max_prefix < 0) return SGL_ERR_INVALID_ARG;
  *empty = batch == 0 || total_extend == 0;
  if (*empty) return SGL_OK;
  if (!kv_fp8 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
    return SGL_ERR_INVALID_ARG;
  if (!q || !pool_k || !pool_v || !req_to_token || !req_pool_idx || !prefix_lens || !extend_lens ||
      !out)
    return SGL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool_k) || !aligned16(pool_v) || !aligned16(out))
    return SGL_ERR_INVALID_ARG;
  if (rtt_rows <= 0 || rtt_stride <= 0 || max_extend > total_extend) return SGL_ERR_INVALID_ARG;
  if (workspace == nullptr || workspace_bytes < extend_workspace_bytes() || !aligned16(workspace))
    return SGL_ERR_WORKSPACE;
  ExtendArgs& a = *ap;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.req_to_token = req_to_token;
  a.rtt_stride = rtt_stride;
  a.req_pool_idx = req_pool_idx;
  a.prefix_lens = prefix_lens;
  a.extend_lens = extend_lens;
  a.batch = batch;
  a.total_extend = total_extend;
  a.max_extend = max_extend;
  a.pool_size = dims->pool_size;
  a.out = out;
  a.workspace = workspace;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.head_dim = dims->head_dim;
  a.sm_scale = scale;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return SGL_OK;
}

sgl_status extend_entry(const void* q, const void* k_new, const void* v_new, const void* pool_k,
                        const void* pool_v, bool kv_fp8, float k_scale, float v_scale,
                        const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                        const int32_t* req_pool_idx, const int32_t* prefix_lens,
                        const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                        int32_t max_extend, int32_t max_prefix, void* out, void* workspace,
                        size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream) {
  ExtendArgs a;
  bool empty = false;
  const sgl_status st = extend_args(q, k_new, v_new, pool_k, pool_v, kv_fp8, k_scale, v_scale, req_to_token,
                                    rtt_rows, rtt_stride, req_pool_idx, prefix_lens, extend_lens, batch,
                                    total_extend, max_extend, max_prefix, out, workspace, workspace_bytes,
                                    dims, &a, &empty);
  if (st != SGL_OK || empty) return st;
  return launch_extend(a, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

sgl_status sgl_extend_attention(const void* q, const void* k_new, const void* v_new,
                                const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                                int32_t max_extend, int32_t max_prefix, void* out, void* workspace,
                                size_t workspace_bytes, const sgl_attn_dims* dims,
                                sgl_stream_t stream) {
  if (batch > 0 && total_extend > 0 && (!k_new || !v_new)) return SGL_ERR_INVALID_ARG;
  return extend_entry(q, k_new, v_new, pool_k, pool_v, false, 1.f, 1.f, req_to_token, rtt_rows,
                      rtt_stride, req_pool_idx, prefix_lens, extend_lens, batch, total_extend,
                      max_extend, max_prefix, out, workspace, workspace_bytes, dims, stream);
}

sgl_status sgl_extend_attention_fp8(const void* q, const void* pool_k, const void* pool_v,
                                    float k_scale, float v_scale, const int32_t* req_to_token,
                                    int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                    const int32_t* extend_lens, int32_t batch,
                                    int32_t total_extend, int32_t max_extend, int32_t max_prefix,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    const sgl_attn_dims* dims, sgl_stream_t stream) {
  if (!valid_kv_scale(k_scale) || !valid_kv_scale(v_scale)) return SGL_ERR_INVALID_ARG;
  return extend_entry(q, nullptr, nullptr, pool_k, pool_v, true, k_scale, v_scale, req_to_token,
                      rtt_rows, rtt_stride, req_pool_idx, prefix_lens, extend_lens, batch,
                      total_extend, max_extend, max_prefix, out, workspace, workspace_bytes, dims,
                      stream);
}

namespace {
sgl_status decode_entry(const void* q, const void* pool_k, const void* pool_v, bool kv_fp8,
                        float k_scale, float v_scale, const int32_t* req_to_token, int32_t rtt_rows,
                        int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
                        int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                        size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream);
}  // namespace

sgl_status sgl_decode_attention(const void* q, const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* seq_lens,
                                int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                                size_t workspace_bytes, const sgl_attn_dims* dims,
                                sgl_stream_t stream) {
  return decode_entry(q, pool_k, pool_v, false, 1.f, 1.f, req_to_token, rtt_rows, rtt_stride,
                      req_pool_idx, seq_lens, batch, max_seq_len, out, workspace, workspace_bytes,
                      dims, stream);
}

sgl_status sgl_decode_attention_fp8(const void* q, const void* pool_k, const void* pool_v,
                                    float k_scale, float v_scale, const int32_t* req_to_token,
                                    int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                                    size_t workspace_bytes, const sgl_attn_dims* dims,
                                    sgl_stream_t stream) {
  if (!valid_kv_scale(k_scale) || !valid_kv_scale(v_scale)) return SGL_ERR_INVALID_ARG;
  return decode_entry(q, pool_k, pool_v, true, k_scale, v_scale, req_to_token, rtt_rows,
                      rtt_stride, req_pool_idx, seq_lens, batch, max_seq_len, out, workspace,
                      workspace_bytes, dims, stream);
}

namespace {
// Host checks of a decode call; fills *a.  *empty: nothing to launch.
sgl_status decode_args(const void* q, const void* pool_k, const void* pool_v, bool kv_fp8,
                       float k_scale, float v_scale, const int32_t* req_to_token, int32_t rtt_rows,
                       int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
                       int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                       size_t workspace_bytes, const sgl_attn_dims* dims, DecodeArgs* ap, bool* empty) {
  float scale;
  const sgl_status st = sgl::validate_decode_call(q, pool_k, pool_v, req_to_token, rtt_rows, rtt_stride,
                                                  req_pool_idx, seq_lens, batch, max_seq_len, out, dims,
                                                  &scale);
  *empty = batch == 0;
  if (st != SGL_OK || *empty) return st;
  const size_t need = decode_workspace_bytes(batch, max_seq_len, dims->num_q_heads,
                                             dims->num_kv_heads, dims->head_dim);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return SGL_ERR_WORKSPACE;
  DecodeArgs& a = *ap;
  a = DecodeArgs{};
  a.q = q;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.req_to_token = req_to_token;
  a.rtt_stride = rtt_stride;
  a.req_pool_idx = req_pool_idx;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq_len = max_seq_len;
  a.out = out;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.head_dim = dims->head_dim;
  a.sm_scale = scale;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return SGL_OK;
}

sgl_status decode_entry(const void* q, const void* pool_k, const void* pool_v, bool kv_fp8,
                        float k_scale, float v_scale, const int32_t* req_to_token, int32_t rtt_rows,
                        int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
                        int32_t batch, int32_t max_seq_len, void* out, void* workspace,
                        size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream) {
  DecodeArgs a;
  bool empty = false;
  const sgl_status st = decode_args(q, pool_k, pool_v, kv_fp8, k_scale, v_scale, req_to_token, rtt_rows,
                                    rtt_stride, req_pool_idx, seq_lens, batch, max_seq_len, out, workspace,
                                    workspace_bytes, dims, &a, &empty);
  if (st != SGL_OK || empty) return st;
  return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

namespace {
sgl_status cascade_entry(
    const void* q, const void* pool_k, const void* pool_v, bool kv_fp8, float k_scale,
    float v_scale, const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
    const int32_t* req_pool_idx, const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
    const int32_t* group_start, const int32_t* group_len, const int32_t* group_depth,
    const int32_t* group_member_off, const int32_t* group_members, int32_t n_groups,
    int32_t max_group_members, int32_t max_depth, void* out, void* workspace,
    size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream) {
  float scale;
  sgl_status st = check_dims(dims, &scale);
  if (st != SGL_OK) return st;
  if (batch < 0 || max_seq_len < 0 || n_groups < 0 || max_group_members < 0 || max_depth < 0)
    return SGL_ERR_INVALID_ARG;
  if (batch == 0) return SGL_OK;
  if (max_seq_len < 1) return SGL_ERR_INVALID_ARG;
  if (!q || !pool_k || !pool_v || !req_to_token || !req_pool_idx || !seq_lens || !out)
    return SGL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool_k) || !aligned16(pool_v)) return SGL_ERR_INVALID_ARG;
  if (rtt_rows <= 0 || rtt_stride <= 0) return SGL_ERR_INVALID_ARG;
  if (n_groups > 0) {
    if (!group_start || !group_len || !group_depth || !group_member_off || !group_members)
      return SGL_ERR_INVALID_ARG;
    if (max_depth < 1 || max_group_members < 1) return SGL_ERR_INVALID_ARG;
    if (n_groups > 65535) return SGL_ERR_UNSUPPORTED;
  }
  const size_t need = decode_workspace_bytes(batch, max_seq_len, dims->num_q_heads,
                                             dims->num_kv_heads, dims->head_dim, true, max_depth);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return SGL_ERR_WORKSPACE;
  DecodeArgs a;
  a.q = q;
  a.pool_k = pool_k;
  a.pool_v = pool_v;
  a.req_to_token = req_to_token;
  a.rtt_stride = rtt_stride;
  a.req_pool_idx = req_pool_idx;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq_len = max_seq_len;
  a.out = out;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.num_q_heads = dims->num_q_heads;
  a.num_kv_heads = dims->num_kv_heads;
  a.head_dim = dims->head_dim;
  a.sm_scale = scale;
  a.cascade = true;
  a.group_start = group_start;
  a.group_len = group_len;
  a.group_depth = group_depth;
  a.group_member_off = group_member_off;
  a.group_members = group_members;
  a.n_groups = n_groups;
  a.max_group_members = max_group_members;
  a.max_depth = max_depth;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}
}  // namespace

sgl_status sgl_cascade_decode_attention(
    const void* q, const void* pool_k, const void* pool_v, const int32_t* req_to_token,
    int32_t rtt_rows, int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
    int32_t batch, int32_t max_seq_len, const int32_t* group_start, const int32_t* group_len,
    const int32_t* group_depth, const int32_t* group_member_off, const int32_t* group_members,
    int32_t n_groups, int32_t max_group_members, int32_t max_depth, void* out, void* workspace,
    size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream) {
  return cascade_entry(q, pool_k, pool_v, false, 1.f, 1.f, req_to_token, rtt_rows, rtt_stride,
                       req_pool_idx, seq_lens, batch, max_seq_len, group_start, group_len,
                       group_depth, group_member_off, group_members, n_groups, max_group_members,
                       max_depth, out, workspace, workspace_bytes, dims, stream);
}

sgl_status sgl_cascade_decode_attention_fp8(
    const void* q, const void* pool_k, const void* pool_v, float k_scale, float v_scale,
    const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
    const int32_t* req_pool_idx, const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
    const int32_t* group_start, const int32_t* group_len, const int32_t* group_depth,
    const int32_t* group_member_off, const int32_t* group_members, int32_t n_groups,
    int32_t max_group_members, int32_t max_depth, void* out, void* workspace,
    size_t workspace_bytes, const sgl_attn_dims* dims, sgl_stream_t stream) {
  if (!valid_kv_scale(k_scale) || !valid_kv_scale(v_scale)) return SGL_ERR_INVALID_ARG;
  return cascade_entry(q, pool_k, pool_v, true, k_scale, v_scale, req_to_token, rtt_rows,
                       rtt_stride, req_pool_idx, seq_lens, batch, max_seq_len, group_start,
                       group_len, group_depth, group_member_off, group_members, n_groups,
                       max_group_members, max_depth, out, workspace, workspace_bytes, dims, stream);
}

size_t sgl_check_cascade_scratch_bytes(int32_t batch, int32_t max_depth) {
  if (batch <= 0 || max_depth <= 0) return 16;
  return ((size_t)batch * (size_t)max_depth * sizeof(int32_t) + 15) / 16 * 16;
}

sgl_status sgl_check_cascade_groups(const int32_t* req_to_token, int32_t rtt_rows,
                                    int32_t rtt_stride, const int32_t* req_pool_idx,
                                    const int32_t* seq_lens, int32_t batch,
                                    const int32_t* group_start, const int32_t* group_len,
                                    const int32_t* group_depth, const int32_t* group_member_off,
                                    const int32_t* group_members, int32_t n_groups,
                                    int32_t max_group_members, int32_t max_depth, void* scratch,
                                    size_t scratch_bytes, int32_t* d_error, sgl_stream_t stream) {
  if (batch < 0 || n_groups < 0 || max_group_members < 0 || max_depth < 0 || rtt_rows <= 0 ||
      rtt_stride <= 0 || d_error == nullptr)
    return SGL_ERR_INVALID_ARG;
  if (batch == 0 || n_groups == 0) return SGL_OK;
  if (!req_to_token || !req_pool_idx || !seq_lens || !group_start || !group_len || !group_depth ||
      !group_member_off || !group_members || max_depth < 1)
    return SGL_ERR_INVALID_ARG;
  const size_t need = sgl_check_cascade_scratch_bytes(batch, max_depth);
  if (scratch == nullptr || scratch_bytes < need) return SGL_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0xFF, need, s) != cudaSuccess) return SGL_ERR_CUDA;
  int32_t* owner = static_cast<int32_t*>(scratch);
  const unsigned blocks = (unsigned)(n_groups < 4096 ? n_groups : 4096);
  check_groups_kernel<<<blocks, 256, 0, s>>>(req_to_token, rtt_rows, rtt_stride, req_pool_idx,
                                             seq_lens, batch, group_start, group_len, group_depth,
                                             group_member_off, group_members, n_groups,
                                             max_group_members, max_depth, owner, d_error);
  check_tiling_kernel<<<(unsigned)((batch + 255) / 256), 256, 0, s>>>(owner, batch, max_depth,
                                                                      group_start, group_len,
                                                                      d_error);
  return last_launch();
}

sgl_status sgl_check_store_kv_indices(const int32_t* slots, int32_t n, int64_t pool_size,
                                      void* bitmap, size_t bitmap_bytes, int32_t* d_error,
                                      sgl_stream_t stream) {
  if (n < 0 || pool_size <= 0 || d_error == nullptr) return SGL_ERR_INVALID_ARG;
  if (n == 0) return SGL_OK;
  if (slots == nullptr) return SGL_ERR_INVALID_ARG;
  const size_t need = (((size_t)pool_size + 31) / 32 * 4 + 15) / 16 * 16;
  if (bitmap == nullptr || bitmap_bytes < need) return SGL_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(bitmap, 0, need, s) != cudaSuccess) return SGL_ERR_CUDA;
  int64_t blocks = ((int64_t)n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  check_store_kernel<<<(unsigned)blocks, 256, 0, s>>>(slots, n, pool_size,
                                                      static_cast<uint32_t*>(bitmap), d_error);
  return last_launch();
}

namespace {
sgl_status check_extend(const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                        const int32_t* req_pool_idx, const int32_t* prefix_lens,
                        const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                        int32_t max_extend, int32_t max_prefix, int64_t pool_size, int32_t* d_error,
                        sgl_stream_t stream, int mode) {
  if (batch < 0 || rtt_rows <= 0 || rtt_stride <= 0 || pool_size <= 0 || d_error == nullptr)
    return SGL_ERR_INVALID_ARG;
  if (batch == 0) return SGL_OK;
  if (!req_to_token || !req_pool_idx || !prefix_lens || !extend_lens) return SGL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  check_rows_kernel<<<(unsigned)batch, 256, 0, s>>>(req_to_token, rtt_rows, rtt_stride, req_pool_idx,
                                                    prefix_lens, extend_lens, mode, pool_size,
                                                    max_prefix, max_extend, d_error);
  check_sum_kernel<<<1, 1024, 0, s>>>(extend_lens, batch, total_extend, d_error);
  return last_launch();
}
}  // namespace

sgl_status sgl_check_extend_indices(const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* prefix_lens,
                                    const int32_t* extend_lens, int32_t batch, int32_t total_extend,
                                    int32_t max_extend, int32_t max_prefix, int64_t pool_size,
                                    int32_t* d_error, sgl_stream_t stream) {
  return check_extend(req_to_token, rtt_rows, rtt_stride, req_pool_idx, prefix_lens, extend_lens,
                      batch, total_extend, max_extend, max_prefix, pool_size, d_error, stream, 0);
}

sgl_status sgl_check_extend_fp8_indices(const int32_t* req_to_token, int32_t rtt_rows,
                                        int32_t rtt_stride, const int32_t* req_pool_idx,
                                        const int32_t* prefix_lens, const int32_t* extend_lens,
                                        int32_t batch, int32_t total_extend, int32_t max_extend,
                                        int32_t max_prefix, int64_t pool_size, int32_t* d_error,
                                        sgl_stream_t stream) {
  return check_extend(req_to_token, rtt_rows, rtt_stride, req_pool_idx, prefix_lens, extend_lens,
                      batch, total_extend, max_extend, max_prefix, pool_size, d_error, stream, 2);
}

sgl_status sgl_check_decode_indices(const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                    const int32_t* req_pool_idx, const int32_t* seq_lens,
                                    int32_t batch, int32_t max_seq_len, int64_t pool_size,
                                    int32_t* d_error, sgl_stream_t stream) {
  if (batch < 0 || rtt_rows <= 0 || rtt_stride <= 0 || pool_size <= 0 || d_error == nullptr)
    return SGL_ERR_INVALID_ARG;
  if (batch == 0) return SGL_OK;
  if (!req_to_token || !req_pool_idx || !seq_lens) return SGL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  check_rows_kernel<<<(unsigned)batch, 256, 0, s>>>(req_to_token, rtt_rows, rtt_stride, req_pool_idx,
                                                    seq_lens, nullptr, 1, pool_size, max_seq_len, 0,
                                                    d_error);
  return last_launch();
}

sgl_status sgl_mixed_attention(
    const void* q_ext, const void* k_new, const void* v_new, const int32_t* ext_req_pool_idx,
    const int32_t* prefix_lens, const int32_t* extend_lens, int32_t ext_batch, int32_t total_extend,
    int32_t max_extend, int32_t max_prefix, void* out_ext, void* ext_workspace, size_t ext_workspace_bytes,
    const void* q_dec, const int32_t* dec_req_pool_idx, const int32_t* seq_lens, int32_t dec_batch,
    int32_t max_seq_len, void* out_dec, void* dec_workspace, size_t dec_workspace_bytes, const void* pool_k,
    const void* pool_v, const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride, int32_t extend_sms,
    const sgl_attn_dims* dims, sgl_stream_t stream) {
  ExtendArgs ea;
  DecodeArgs da;
  bool e_empty = true, d_empty = true;
  sgl_status st = extend_args(q_ext, k_new, v_new, pool_k, pool_v, false, 1.f, 1.f, req_to_token, rtt_rows,
                              rtt_stride, ext_req_pool_idx, prefix_lens, extend_lens, ext_batch, total_extend,
                              max_extend, max_prefix, out_ext, ext_workspace, ext_workspace_bytes, dims, &ea,
                              &e_empty);
  if (st != SGL_OK) return st;
  st = decode_args(q_dec, pool_k, pool_v, false, 1.f, 1.f, req_to_token, rtt_rows, rtt_stride,
                   dec_req_pool_idx, seq_lens, dec_batch, max_seq_len, out_dec, dec_workspace,
                   dec_workspace_bytes, dims, &da, &d_empty);
  if (st != SGL_OK) return st;
  if (e_empty) ea.batch = 0;
  if (d_empty) da.batch = 0;
  if (extend_sms < 0) return SGL_ERR_INVALID_ARG;
  if (extend_sms == 0 && !e_empty && !d_empty) {
    // split the SMs by an estimate of each side's time from the host values
    // (mean lengths taken as half the maxima): extend flops at ~1.2 PFLOP/s,
    // decode bytes at ~6.7 TB/s; CTAs whose side finishes first take the
    // other side's work, so the estimate only sets where both start
    const double te = 4.0 * dims->head_dim * dims->num_q_heads * (double)total_extend *
                      (0.5 * max_prefix + 0.5 * max_extend) / 1.2e15;
    const double td = (double)dec_batch * 0.5 * max_seq_len *
                      (4.0 * dims->num_kv_heads * dims->head_dim + 4.0) / 6.7e12;
    const int n = num_sms();
    extend_sms = (int32_t)(n * te / (te + td) + 0.5);
    if (extend_sms < 1) extend_sms = 1;
    if (extend_sms > n - 1) extend_sms = n - 1;
  }
  return launch_mixed(ea, da, extend_sms, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
