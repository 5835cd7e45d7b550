// store_kv: scatter new K/V rows into their pool slots (bit-exact copy).
//
// "Origins: the paper and the first commit", Execution: RadixAttention and
// two sets of kernels -- store_kv_cache assigns the layer's new keys and
// values into the key and value buffers at out_cache_loc.
//
// One warp moves one (token, K or V) row: all Hkv heads of a slot are
// contiguous (Hkv * D * 2 bytes: 2 KiB for 8 heads of 128), so each row is
// one coalesced 16-byte-per-lane read and one coalesced write.  HBM-bound for
// large batches (read 2 rows + write 2 rows per token), launch-bound for small.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace sgl {

namespace {

constexpr int kStoreWarps = 8;

SGL_DEV uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kStoreWarps * 32)
store_kv_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                const int32_t* __restrict__ slots, int32_t n, uint4* __restrict__ pool_k,
                uint4* __restrict__ pool_v, int32_t row_vecs) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
  const int64_t total_rows = 2 * (int64_t)n;
  const int64_t nwarps = (int64_t)gridDim.x * kStoreWarps;
  for (int64_t row = warp; row < total_rows; row += nwarps) {
    const bool is_v = row >= n;
    const int64_t i = is_v ? row - n : row;
    const int64_t slot = slots[i];
    const uint4* src = (is_v ? v_new : k_new) + i * row_vecs;
    uint4* dst = (is_v ? pool_v : pool_k) + slot * row_vecs;
    // up to 4 outstanding 16-byte loads per lane before the stores
    int c = lane;
    for (; c + 96 < row_vecs; c += 128) {
      uint4 a = ld_stream(src + c), b = ld_stream(src + c + 32);
      uint4 d = ld_stream(src + c + 64), e = ld_stream(src + c + 96);
      dst[c] = a;
      dst[c + 32] = b;
      dst[c + 64] = d;
      dst[c + 96] = e;
    }
    for (; c < row_vecs; c += 32) dst[c] = ld_stream(src + c);
  }
}

// FP8 pool: a warp quantises one (token, K or V) row.  Each lane turns two
// 16-byte vectors of bf16 into one 16-byte vector of e4m3 codes:
// code = e4m3(x / scale), the quotient in IEEE float32 and the conversion to
// nearest (ties to even), saturating to +-448 ("Inside SGLang", Step 6:
// --kv-cache-dtype fp8_e4m3 with per-tensor scales from the checkpoint).
SGL_DEV uint32_t quant4(uint32_t lo, uint32_t hi, float scale) {
  auto q2 = [&](uint32_t w) {
    const float a = __fdiv_rn(__uint_as_float(w << 16), scale);
    const float b = __fdiv_rn(__uint_as_float(w & 0xFFFF0000u), scale);
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  };
  return q2(lo) | (q2(hi) << 16);
}

__global__ void __launch_bounds__(kStoreWarps * 32)
store_kv_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                    const int32_t* __restrict__ slots, int32_t n, uint4* __restrict__ pool_k,
                    uint4* __restrict__ pool_v, int32_t out_vecs, float k_scale, float v_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
  const int64_t total_rows = 2 * (int64_t)n;
  const int64_t nwarps = (int64_t)gridDim.x * kStoreWarps;
  for (int64_t row = warp; row < total_rows; row += nwarps) {
    const bool is_v = row >= n;
    const int64_t i = is_v ? row - n : row;
    const int64_t slot = slots[i];
    const float scale = is_v ? v_scale : k_scale;
    const uint4* src = (is_v ? v_new : k_new) + i * 2 * out_vecs;
    uint4* dst = (is_v ? pool_v : pool_k) + slot * out_vecs;
    for (int c = lane; c < out_vecs; c += 32) {
      const uint4 a = ld_stream(src + 2 * c), b = ld_stream(src + 2 * c + 1);
      dst[c] = make_uint4(quant4(a.x, a.y, scale), quant4(a.z, a.w, scale), quant4(b.x, b.y, scale),
                          quant4(b.z, b.w, scale));
    }
  }
}

}  // namespace

sgl_status launch_store_kv_fp8(const void* k_new, const void* v_new, const int32_t* slots,
                               int32_t n, void* pool_k, void* pool_v, int32_t row_elems,
                               float k_scale, float v_scale, cudaStream_t stream) {
  if (n == 0) return SGL_OK;
  const int32_t out_vecs = row_elems / 16;
  const int64_t rows = 2 * (int64_t)n;
  int64_t blocks = (rows + kStoreWarps - 1) / kStoreWarps;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  store_kv_fp8_kernel<<<(unsigned)blocks, kStoreWarps * 32, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, n,
      static_cast<uint4*>(pool_k), static_cast<uint4*>(pool_v), out_vecs, k_scale, v_scale);
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

sgl_status launch_store_kv(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                           void* pool_k, void* pool_v, int32_t row_bytes, cudaStream_t stream) {
  if (n == 0) return SGL_OK;
  const int32_t row_vecs = row_bytes / 16;
  const int64_t rows = 2 * (int64_t)n;
  int64_t blocks = (rows + kStoreWarps - 1) / kStoreWarps;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  store_kv_kernel<<<(unsigned)blocks, kStoreWarps * 32, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slots, n,
      static_cast<uint4*>(pool_k), static_cast<uint4*>(pool_v), row_vecs);
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

}  // namespace sgl
