// Launchers of the extend and cascade-group kernels (extend_dev.cuh): host
// checks of the shapes the kernels are built for, grid sizes and parameters.
#include "extend_dev.cuh"
#include "launch.h"

namespace sgl {

using namespace ext;

namespace {

template <int D, bool kFp8>
sgl_status run(const Params& prm, int32_t batch, int32_t max_extend, cudaStream_t stream) {
  constexpr int kThreads = Roles<kFp8>::kThreads;
  constexpr int kSmem = smem_bytes<D, kFp8>();
  auto kern = extend_kernel<D, kFp8>;
  if (kernel_blocks_per_sm<extend_kernel<D, kFp8>>(kSmem, kThreads) < 0) return SGL_ERR_CUDA;
  if (Roles<kFp8>::kSplitRegs && !kernel_regs_at_least<extend_kernel<D, kFp8>>(Roles<kFp8>::kLaunchRegs))
    return SGL_ERR_UNSUPPORTED;
  const int per_cta = 2 * prm.tpt;
  const unsigned gx = (unsigned)((max_extend + per_cta - 1) / per_cta);
  dim3 grid(gx, (unsigned)prm.Hkv, (unsigned)batch);
  kern<<<grid, kThreads, kSmem, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

template <int D, bool kFp8>
sgl_status run_groups(const Params& prm, int32_t n_groups, int32_t max_members, cudaStream_t stream,
                      bool dependent) {
  // bf16 pools: one Q tile a CTA, two CTAs an SM (most groups of a tree fill
  // one tile; the second CTA's work hides each CTA's start and end)
  constexpr int kTiles = kFp8 ? 2 : kGroupTilesBf16;
  constexpr int kThreads = Roles<kFp8, kTiles>::kThreads;
  constexpr int kSmem = smem_bytes<D, kFp8, kTiles>();
  auto kern = cascade_group_kernel<D, kFp8, kTiles>;
  if (kernel_blocks_per_sm<cascade_group_kernel<D, kFp8, kTiles>>(kSmem, kThreads) < 0) return SGL_ERR_CUDA;
  if (Roles<kFp8, kTiles>::kSplitRegs &&
      !kernel_regs_at_least<cascade_group_kernel<D, kFp8, kTiles>>(Roles<kFp8, kTiles>::kLaunchRegs))
    return SGL_ERR_UNSUPPORTED;
  const int per_cta = kTiles * prm.tpt;
  const unsigned gx = (unsigned)((max_members + per_cta - 1) / per_cta);
  dim3 grid(gx, (unsigned)prm.Hkv, (unsigned)n_groups);
  if (dependent) {
    if (launch_dependent(kern, grid, dim3(kThreads), kSmem, stream, prm) != cudaSuccess) return SGL_ERR_CUDA;
  } else {
    kern<<<grid, kThreads, kSmem, stream>>>(prm);
  }
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

template <bool kFp8>
sgl_status dispatch(int head_dim, bool groups, const Params& prm, int32_t n, int32_t max_rows,
                    cudaStream_t stream, bool dependent = false) {
  if (head_dim == 128)
    return groups ? run_groups<128, kFp8>(prm, n, max_rows, stream, dependent)
                  : run<128, kFp8>(prm, n, max_rows, stream);
  if (head_dim == 64)
    return groups ? run_groups<64, kFp8>(prm, n, max_rows, stream, dependent)
                  : run<64, kFp8>(prm, n, max_rows, stream);
  return SGL_ERR_UNSUPPORTED;
}

}  // namespace

sgl_status launch_cascade_groups(const GroupArgs& a, cudaStream_t stream, bool dependent) {
  if (a.n_groups == 0 || a.max_members == 0) return SGL_OK;
  const int g = a.num_q_heads / a.num_kv_heads;
  if (g < 1 || g > BM) return SGL_ERR_UNSUPPORTED;
  if (a.n_groups > 65535 || a.num_kv_heads > 65535) return SGL_ERR_UNSUPPORTED;
  Params prm = {};
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.pool_k = static_cast<const __nv_bfloat16*>(a.pool_k);
  prm.pool_v = static_cast<const __nv_bfloat16*>(a.pool_v);
  prm.pool_k8 = static_cast<const uint8_t*>(a.pool_k);
  prm.pool_v8 = static_cast<const uint8_t*>(a.pool_v);
  prm.req_to_token = a.req_to_token;
  prm.rtt_stride = a.rtt_stride;
  prm.req_pool_idx = a.req_pool_idx;
  prm.Hq = a.num_q_heads;
  prm.Hkv = a.num_kv_heads;
  prm.g = g;
  prm.tpt = BM / g;
  prm.rows_used = prm.tpt * g;
  // e4m3: scores in units of the widened codes (code * 2^-8) times the K
  // scale; the states' P.V rows are left in code units (the decode combine
  // applies the V scale)
  prm.scale_log2 = a.sm_scale * 1.4426950408889634f * (a.kv_fp8 ? a.k_scale * kFp8Operand : 1.f);
  prm.o_scale = a.kv_fp8 ? kFp8Operand : 1.f;
  prm.status = a.status;
  prm.wait_ns = device_wait_limit_ns();
  prm.group_start = a.group_start;
  prm.group_len = a.group_len;
  prm.group_depth = a.group_depth;
  prm.member_off = a.member_off;
  prm.members = a.members;
  prm.part_ml = static_cast<float2*>(a.part_ml);
  prm.part_acc = static_cast<float*>(a.part_acc);
  prm.part_base = a.part_base;
  prm.max_depth = a.max_depth;
  prm.batch = a.batch;
  return a.kv_fp8 ? dispatch<true>(a.head_dim, true, prm, a.n_groups, a.max_members, stream, dependent)
                  : dispatch<false>(a.head_dim, true, prm, a.n_groups, a.max_members, stream, dependent);
}

size_t extend_workspace_bytes() { return 256; }

sgl_status launch_extend(const ExtendArgs& a, cudaStream_t stream) {
  if (a.batch == 0 || a.total_extend == 0 || a.max_extend == 0) return SGL_OK;
  Params prm;
  const sgl_status st = make_extend_params(a, &prm);
  if (st != SGL_OK) return st;
  return a.kv_fp8 ? dispatch<true>(a.head_dim, false, prm, a.batch, a.max_extend, stream)
                  : dispatch<false>(a.head_dim, false, prm, a.batch, a.max_extend, stream);
}

}  // namespace sgl
