// Launchers of the decode kernels (decode_dev.cuh): the workspace layout,
// shape checks, the plan / split / combine launches and the cascade's group
// pass before the split.
#include "decode_dev.cuh"
#include "launch.h"

namespace sgl {

using namespace dec;

namespace {

template <int D, int G, typename KV>
sgl_status run(const Params& prm, int64_t max_items, const Groups& gr, const GroupArgs* ga,
               cudaStream_t stream) {
  constexpr int LPT = (D == 128 && G >= 4) ? 16 : 8;
  constexpr size_t kRing = SplitRing<KV, G>::template bytes<D>();
  constexpr size_t smem = kRing + kItemMax * sizeof(int32_t);
  static_assert(kWarps * G * (D + 2) * sizeof(float) <= kRing, "reduction scratch must fit in the ring");
  // e4m3 pools: a slot's rows of kWarps adjacent KV heads gathered as one span
  // (spans_for)
  constexpr bool kFp8 = sizeof(KV) == 1;
  const bool spans = kFp8 && spans_for(prm.Hkv, prm.kv_split, true);
  auto kern = decode_split_kernel<D, G, LPT, KV, false>;
  int blocks_per_sm;
  if constexpr (kFp8) {
    if (spans) kern = decode_split_kernel<D, G, LPT, KV, true>;
    blocks_per_sm = spans ? kernel_blocks_per_sm<decode_split_kernel<D, G, LPT, KV, true>>((int)smem, kThreads)
                          : kernel_blocks_per_sm<decode_split_kernel<D, G, LPT, KV, false>>((int)smem, kThreads);
  } else {
    blocks_per_sm = kernel_blocks_per_sm<decode_split_kernel<D, G, LPT, KV, false>>((int)smem, kThreads);
  }
  if (blocks_per_sm < 0) return SGL_ERR_CUDA;
  const int gy = spans ? prm.Hkv / kWarps : prm.Hkv;  // grid y: counters (heads or head groups)
  // plan, split kernel, the cascade's group pass, combine: each launched
  // dependent on the one before (it may start while that one runs, and
  // waits for what it needs); the group pass reads nothing of the split
  // kernel's and fills the SMs the split kernel's last units leave
  decode_plan_kernel<<<1, 1024, 0, stream>>>(prm.seq_lens, prm.batch, max_items, prm.chunk, prm.Hkv, prm.ws,
                                             gr);
  // one wave of resident CTAs, every CTA taking items while any are left
  // (measured against two waves: tree cascade +5.5%, Llama-7B-like decode
  // +1.8%, chunked-mix decode kernel +1.2%)
  int64_t gx = ((int64_t)blocks_per_sm * num_sms() + gy - 1) / gy;
  if (gx > max_items) gx = max_items;
  if (gx < 1) gx = 1;
  if (launch_dependent(kern, dim3((unsigned)gx, (unsigned)gy), dim3(kThreads), smem, stream, prm) != cudaSuccess)
    return SGL_ERR_CUDA;
  if (ga != nullptr) {
    const sgl_status st = launch_cascade_groups(*ga, stream, true);
    if (st != SGL_OK) return st;
  }
  const int64_t warps = (int64_t)prm.batch * prm.Hq;
  if (launch_dependent(decode_combine_kernel<D>, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0, stream, prm) !=
      cudaSuccess)
    return SGL_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

template <int D, typename KV>
sgl_status run_g(int G, const Params& prm, int64_t max_items, const Groups& gr,
                 const GroupArgs* ga, cudaStream_t stream) {
  switch (G) {
    case 1: return run<D, 1, KV>(prm, max_items, gr, ga, stream);
    case 2: return run<D, 2, KV>(prm, max_items, gr, ga, stream);
    case 4: return run<D, 4, KV>(prm, max_items, gr, ga, stream);
    case 8: return run<D, 8, KV>(prm, max_items, gr, ga, stream);
    case 3: return run<D, 3, KV>(prm, max_items, gr, ga, stream);
    case 5: return run<D, 5, KV>(prm, max_items, gr, ga, stream);
    case 6: return run<D, 6, KV>(prm, max_items, gr, ga, stream);
    case 7: return run<D, 7, KV>(prm, max_items, gr, ga, stream);
    case 9: return run<D, 9, KV>(prm, max_items, gr, ga, stream);
    case 10: return run<D, 10, KV>(prm, max_items, gr, ga, stream);
    case 11: return run<D, 11, KV>(prm, max_items, gr, ga, stream);
    case 12: return run<D, 12, KV>(prm, max_items, gr, ga, stream);
    case 13: return run<D, 13, KV>(prm, max_items, gr, ga, stream);
    case 14: return run<D, 14, KV>(prm, max_items, gr, ga, stream);
    case 15: return run<D, 15, KV>(prm, max_items, gr, ga, stream);
    case 16: return run<D, 16, KV>(prm, max_items, gr, ga, stream);
    default: return SGL_ERR_UNSUPPORTED;
  }
}

}  // namespace

size_t decode_workspace_bytes(int32_t batch, int32_t max_seq_len, int32_t Hq, int32_t Hkv,
                              int32_t D, bool cascade, int32_t max_depth) {
  const size_t head = cascade ? kCascadeStatusBytes : 0;
  if (batch <= 0 || max_seq_len <= 0 || Hkv <= 0 || Hq < Hkv) return head + 256;
  const int32_t split = kv_split_for(Hq / Hkv);
  const int32_t chunk = chunk_for(spans_possible(Hkv * split, split));
  return head + ws_layout(batch, max_items_for(batch, max_seq_len, chunk), Hkv * split, Hq / Hkv / split, D,
                          cascade ? max_depth : 0, cascade, nullptr, nullptr);
}

sgl_status decode_shape_supported(int32_t num_q_heads, int32_t num_kv_heads) {
  if (num_kv_heads <= 0) return SGL_ERR_UNSUPPORTED;
  const int G_pool = num_q_heads / num_kv_heads;
  if (G_pool < 1 || G_pool > 128) return SGL_ERR_UNSUPPORTED;
  // KV heads as the kernels see them: grid y
  if ((int64_t)num_kv_heads * kv_split_for(G_pool) > 65535) return SGL_ERR_UNSUPPORTED;
  return SGL_OK;
}

sgl_status launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch == 0) return SGL_OK;
  if (decode_shape_supported(a.num_q_heads, a.num_kv_heads) != SGL_OK) return SGL_ERR_UNSUPPORTED;
  Params prm;
  DecodePlan pl;
  const sgl_status st = make_decode_params(a, &prm, &pl);
  if (st != SGL_OK) return st;
  const int G = pl.G;
  const int64_t max_items = pl.max_items;
  const Groups& gr = pl.gr;
  const GroupArgs* gp = pl.groups ? &pl.ga : nullptr;
  if (a.kv_fp8) {
    if (a.head_dim == 128) return run_g<128, uint8_t>(G, prm, max_items, gr, gp, stream);
    if (a.head_dim == 64) return run_g<64, uint8_t>(G, prm, max_items, gr, gp, stream);
    return SGL_ERR_UNSUPPORTED;
  }
  if (a.head_dim == 128) return run_g<128, __nv_bfloat16>(G, prm, max_items, gr, gp, stream);
  if (a.head_dim == 64) return run_g<64, __nv_bfloat16>(G, prm, max_items, gr, gp, stream);
  return SGL_ERR_UNSUPPORTED;
}

}  // namespace sgl
