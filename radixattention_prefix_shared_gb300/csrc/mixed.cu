// One launch for a mixed batch: the extend chunks and the decode requests of
// one serving step, over the same pools ("Inside SGLang", Step 10: Split long
// prompts into chunks -- a chunk's prefill and the running requests' decode
// share a forward pass; "A walkthrough of SGLang", the MIXED forward mode).
//
// Extend attention is bound by the tensor cores and decode attention by HBM
// bandwidth, but an extend CTA fills an SM (shared memory, registers, all of
// TMEM), so the two can only overlap by sharing the SMs out.  Here one
// persistent CTA runs on every SM and takes a role ticket when it starts: the
// first extend_ctas tickets take extend tiles (request, KV head, pair of Q
// tiles) from one counter, the others decode work units (item, KV head) from
// another.  A CTA whose queue has run dry takes the other queue's work, so
// both finish together whatever the split.  The extend role runs the extend
// kernel's pipeline tile after tile (attend_tiles in persistent mode: TMEM
// held for the whole launch, barriers invalidated and initialised again for
// every tile); the decode role runs five independent 4-warp groups (a named
// barrier and a ring each) through the split kernel's work loop.  The decode
// plan (work items, and the counters zeroed) runs before and the combine after,
// as for a decode call.  The extend rows and the decode rows are those the
// extend and decode kernels compute: the same code on the same tiles and items.
#include "decode_dev.cuh"
#include "extend_dev.cuh"
#include "launch.h"

namespace sgl {
namespace {

constexpr int kMixThreads = 640;  // 20 warps: the extend roles' 19, in whole warpgroups
// 4-warp decode groups a CTA, and their ring depth: five groups of four
// stages fit below the extend barriers (the split kernel runs four CTAs of
// six stages an SM).  Measured on the chunked-prefill mix's decode batch:
// five groups of four stages 1.41 ms, four of five 1.55 ms, the split kernel
// alone 1.36 ms -- the warps that issue the gathers count more than the
// stages in flight.
constexpr int kDecGroups = 5;
constexpr int kDecDepth = 4;

struct MixParams {
  ext::Params e;
  dec::Params d;
  int32_t e_gx;         // extend tiles along x (pairs of Q tiles of one request)
  int32_t e_tiles;      // extend tiles in all: e_gx * Hkv * batch
  int32_t extend_ctas;  // CTAs that start on extend tiles
  int32_t* counters;    // role tickets, next extend tile, next decode unit
};

// shared memory of one decode group: its ring and slot run (1024-aligned)
template <int D, int G>
constexpr int dec_group_bytes() {
  using Ring = dec::SplitRing<__nv_bfloat16, G>;
  constexpr size_t ring = (size_t)kDecDepth * 2 * Ring::kTileB * D * 2;
  static_assert(dec::kWarps * G * (D + 2) * sizeof(float) <= ring, "reduction scratch fits in the ring");
  return (int)((ring + dec::kItemMax * sizeof(int32_t) + 1023) / 1024 * 1024);
}

// the decode state must fit the extend roles' register budget (96 a thread):
// built for one and two query heads per KV head (the CUDA-core rows)
template <int G>
constexpr bool mixed_decode_built() {
  return G == 1 || G == 2;
}

template <int D, int G, int LPT>
__global__ void __launch_bounds__(kMixThreads, 1) mixed_kernel(MixParams mp) {
  using C = ext::Cfg<D, false>;
  using R = ext::Roles<false>;
  constexpr uint32_t kCols = ext::tmem_cols<2>();
  static_assert(kDecGroups * dec_group_bytes<D, G>() <= (2 + C::kStages) * C::kTileBytes,
                "the decode rings end below the extend barriers");
  static_assert(R::kThreads <= kMixThreads && kDecGroups * dec::kThreads <= kMixThreads, "roles");
  uint8_t* smem = ext::smem_base();
  ext::Bars* bars = ext::bars_of<D, false, 2>(smem);
  __shared__ int32_t s_ticket, s_tile;
  __shared__ int32_t s_item[kDecGroups][2];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    ext::init_barriers_once<C::kStages>(bars);
    bars->abort = 0;
    s_ticket = atomicAdd(&mp.counters[0], 1);
    mbar_fence_init();
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool extend_first = s_ticket < mp.extend_ctas;
  const int32_t hkv_d = mp.d.Hkv;
  const int32_t n_units = *mp.d.ws.n_items * hkv_d;
  bool failed = false;
  for (int pass = 0; pass < 2 && !failed; ++pass) {
    if ((pass == 0) == extend_first) {
      // ---- extend tiles, in the extend grid's order (x fastest)
      for (;;) {
        if (tid == 0) s_tile = atomicAdd(&mp.counters[1], 1);
        __syncthreads();
        const int32_t tile = s_tile;
        __syncthreads();  // every thread has read the index before it is taken again
        if (tile >= mp.e_tiles) break;
        const int32_t per_z = mp.e_gx * mp.e.Hkv;
        ext::attend_tiles<D, false, false, 2, true>(mp.e, tile % mp.e_gx, (tile / mp.e_gx) % mp.e.Hkv,
                                                    tile / per_z);
        // a bounded wait gave up (its status is recorded): this CTA's
        // barriers are no longer in step, so it takes no more work
        if (bars->abort) {
          failed = true;
          break;
        }
      }
    } else {
      // ---- decode units u: item u / Hkv, KV head u % Hkv (the heads of an
      // item run side by side and read the same slots)
      if (warp < 4 * kDecGroups) {
        const int g = warp >> 2;
        dec::split_units<D, G, LPT, __nv_bfloat16, kDecDepth>(
            mp.d, smem + g * dec_group_bytes<D, G>(), s_item[g], tid - dec::kThreads * g, n_units,
            [g] { named_bar_sync(9 + g, dec::kThreads); }, [&] { return atomicAdd(&mp.counters[2], 1); },
            [hkv_d](int32_t u) { return (int)(u % hkv_d); }, [hkv_d](int32_t u) { return u / hkv_d; });
      }
      __syncthreads();  // the rings are free before the extend role reuses the memory
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kCols);
  }
}

template <int D, int G>
sgl_status run_mixed(const MixParams& mp, int64_t max_items, cudaStream_t stream) {
  constexpr int LPT = 8;  // the split kernel's lanes a key at these group sizes
  static_assert(mixed_decode_built<G>(), "decode group size");
  constexpr int kSmem = ext::smem_bytes<D, false>();
  if (kernel_blocks_per_sm<mixed_kernel<D, G, LPT>>(kSmem, kMixThreads) < 0) return SGL_ERR_CUDA;
  dec::decode_plan_kernel<<<1, 1024, 0, stream>>>(mp.d.seq_lens, mp.d.batch, max_items, mp.d.chunk, mp.d.Hkv,
                                                  mp.d.ws, dec::Groups{}, mp.counters);
  mixed_kernel<D, G, LPT><<<(unsigned)num_sms(), kMixThreads, kSmem, stream>>>(mp);
  const int64_t warps = (int64_t)mp.d.batch * mp.d.Hq;
  dec::decode_combine_kernel<D><<<(unsigned)((warps + 3) / 4), 128, 0, stream>>>(mp.d);
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

}  // namespace

bool mixed_launch_built(const ExtendArgs& e, const DecodeArgs& d) {
  if (e.kv_fp8 || d.kv_fp8 || d.cascade) return false;
  if (e.head_dim != d.head_dim || (e.head_dim != 64 && e.head_dim != 128)) return false;
  if (e.num_kv_heads <= 0 || d.num_kv_heads <= 0) return false;
  const int gd = d.num_q_heads / d.num_kv_heads;
  return gd == 1 || gd == 2;
}

sgl_status launch_mixed(const ExtendArgs& ea, const DecodeArgs& da, int32_t extend_ctas,
                        cudaStream_t stream) {
  const bool has_e = ea.batch > 0 && ea.total_extend > 0 && ea.max_extend > 0;
  const bool has_d = da.batch > 0;
  if (!has_e && !has_d) return SGL_OK;
  if (!has_d) return launch_extend(ea, stream);
  if (!has_e) return launch_decode(da, stream);
  if (!mixed_launch_built(ea, da)) {
    // shapes the single launch is not built for: the two kernels in turn
    const sgl_status st = launch_extend(ea, stream);
    return st != SGL_OK ? st : launch_decode(da, stream);
  }
  MixParams mp = {};
  sgl_status st = ext::make_extend_params(ea, &mp.e);
  if (st != SGL_OK) return st;
  dec::DecodePlan pl;
  st = dec::make_decode_params(da, &mp.d, &pl);
  if (st != SGL_OK) return st;
  const int per_cta = 2 * mp.e.tpt;
  mp.e_gx = (ea.max_extend + per_cta - 1) / per_cta;
  const int64_t tiles = (int64_t)mp.e_gx * ea.num_kv_heads * ea.batch;
  if (tiles > INT32_MAX) return SGL_ERR_UNSUPPORTED;
  mp.e_tiles = (int32_t)tiles;
  const int n_sms = num_sms();
  mp.extend_ctas = extend_ctas < 0 ? 0 : (extend_ctas > n_sms ? n_sms : extend_ctas);
  // words 1.. of the extend workspace (word 0 is its status)
  mp.counters = static_cast<int32_t*>(ea.workspace) + 1;
  if (pl.G == 1) {
    return da.head_dim == 128 ? run_mixed<128, 1>(mp, pl.max_items, stream) : run_mixed<64, 1>(mp, pl.max_items, stream);
  }
  return da.head_dim == 128 ? run_mixed<128, 2>(mp, pl.max_items, stream) : run_mixed<64, 2>(mp, pl.max_items, stream);
}

}  // namespace sgl
