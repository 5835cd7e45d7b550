// Extend attention on tcgen05 tensor cores: the new suffix tokens of each
// request attend to the request's cached prefix (gathered from the pool
// through req_to_token) and causally to the suffix itself.
//
// What is computed ("Inside SGLang", Step 3: Look inside the forward pass;
// "Origins: the paper and the first commit", Batching and Execution): for
// suffix query i of a request with prefix length p, scores against keys
// 0..p+i scaled by 1/sqrt(D), softmax, times V -- the last rows of full
// causal attention over prefix+suffix, without recomputing or copying the
// prefix.
//
// Work decomposition: one CTA per (request, KV head, block of 2*tpt suffix
// tokens).  The g = Hq/Hkv query heads that share the KV head are packed into
// the M dimension: row m of a 128-row Q tile is token m/g, head m%g, so every
// gathered K/V row feeds all heads of its group.  The CTA owns two Q tiles
// and walks the KV blocks (128 keys each): first the prefix blocks (rows
// gathered from the pool), then the suffix blocks (rows of k_new/v_new).
//
// Warp roles (11 warps):
//   warps 0-3  softmax for Q tile 0 (TMEM lanes 0-127)
//   warps 4-7  softmax for Q tile 1
//   warps 8-9  producers: 16-byte cp.async gathers of Q, K and V rows into
//              the 128-byte-swizzled shared-memory layout the tensor core reads
//   warp 10    TMEM allocation and the single thread that issues tcgen05.mma
// TMEM (512 columns): S0 | S1 | O0 | O1.  S_t = Q_t K^T lands in TMEM as
// fp32; the softmax warps read it, write P = exp2(S*scale*log2e - m) as
// bf16 over the first half of S_t's columns, and O_t += P V is issued with A
// read from TMEM.  The two Q tiles ping-pong: while softmax works on one
// tile the tensor core computes the other.  The running max is only moved
// when a block's max exceeds it by more than 2^8 (O is then rescaled in
// TMEM), so most blocks need no correction pass.
//
// Every wait on an mbarrier is bounded (2 s); on a timeout the kernel raises
// an abort flag, records a status word in the workspace, drains its own
// in-flight copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "launch.h"

namespace sgl {

namespace {

constexpr int BM = 128;  // rows per Q tile
constexpr int BN = 128;  // keys per KV block
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarps = 2;
constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;  // 10
constexpr int kThreads = (kMmaWarp + 1) * 32;              // 352
constexpr int kProducerThreads = kProducerWarps * 32;
// a producer thread copies 16-byte chunk (ptid % 8) of rows
// ptid / 8 + kRowStep * i, i < kRowsPerThread, of every 128-row tile
constexpr int kRowStep = kProducerThreads / 8;
constexpr int kRowsPerThread = 128 / kRowStep;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTmemCols = 512;
// TMEM column of S_t and O_t
SGL_DEV constexpr uint32_t col_s(int t) { return 128u * t; }
SGL_DEV constexpr uint32_t col_o(int t) { return 256u + 128u * t; }
constexpr int kLag = 2;  // cp.async groups a producer keeps in flight before publishing

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;            // 128-byte column chunks per row
  static constexpr int kChunkBytes = 128 * 128;     // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;    // Q tile or one K / V block
  static constexpr int kStages = D == 128 ? 4 : 8;  // K/V ring slots
  static constexpr int kSmemBytes = (2 + kStages) * kTileBytes + 1024 + 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done;
  uint64_t drain;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint32_t tmem_base;
  int abort;
  int32_t red[32];
};

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* pool_k;
  const __nv_bfloat16* pool_v;
  const int32_t* req_to_token;
  int64_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* prefix_lens;
  const int32_t* extend_lens;
  __nv_bfloat16* out;
  int32_t Hq, Hkv, g, tpt, rows_used;
  float scale_log2;
  int* status;
};

// byte offset of 16-byte chunk `ci` (0..7) of row `row` inside one
// 128-row x 128-byte swizzled chunk
SGL_DEV uint32_t sw128(int row, int ci) { return row * 128 + ((ci ^ (row & 7)) << 4); }

// Warp-collective bounded wait: lane 0 polls, the verdict is broadcast.
SGL_DEV bool warp_wait(uint64_t* bar, uint32_t parity, Bars* bars, int* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, &bars->abort, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) extend_kernel(Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * C::kTileBytes;
  Bars* bars = reinterpret_cast<Bars*>(sKV + C::kStages * C::kTileBytes);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = blockIdx.z, kvh = blockIdx.y;
  const int e = p.extend_lens[r];
  const int q0 = blockIdx.x * 2 * p.tpt;  // first suffix token of this CTA
  if (q0 >= e) return;                    // nothing to do (uniform across the CTA)
  const int pfx = p.prefix_lens[r];
  const int q_end = min(e, q0 + 2 * p.tpt);
  const int nb_pre = (pfx + BN - 1) / BN;
  const int nb = nb_pre + (q_end + BN - 1) / BN;

  // exclusive prefix sum of extend_lens: where request r's rows start
  {
    int32_t part = 0;
    for (int i = tid; i < r; i += kThreads) part += p.extend_lens[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) bars->red[warp] = part;
  }
  if (tid == 0) {
    mbar_init(&bars->q_full, kProducerThreads);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_ready[t], 128);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], kProducerThreads);
      mbar_init(&bars->kv_empty[s], 1);
    }
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  int32_t off = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) off += bars->red[w];
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sQ_a = smem_u32(sQ), sKV_a = smem_u32(sKV);

  if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(t);
    const uint32_t tO = tmem + lane_off + col_o(t);
    const int tok = q0 + t * p.tpt + row / p.g;
    const bool row_valid = row < p.rows_used && tok < e;
    const int tok_i = row_valid ? tok : (1 << 30);  // padding rows see every key
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int b = 0; b < nb && ok; ++b) {
      ok = warp_wait(&bars->s_full[t], b & 1, bars, p.status);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[BN];
#pragma unroll
      for (int j = 0; j < BN / 32; ++j)
        tmem_ld32(tS + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * j]));
      tmem_wait_ld();
      // visible keys of this block: c < limit
      int limit;
      if (b < nb_pre) limit = pfx - b * BN;
      else limit = tok_i - (b - nb_pre) * BN + 1;
      limit = max(0, min(BN, limit));
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        float v = c < limit ? __uint_as_float(sr[c]) : -INFINITY;
        sr[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
      const float mx2 = mx * p.scale_log2;
      const bool need = mx2 > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mx2);
        m_ref = mx2;
      }
      l *= alpha;
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
      float sum = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // keys 64*half .. 64*half+63 -> 32 packed bf16 pairs -> TMEM columns 32*half..
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int k = 64 * half + 2 * c;
          const float p0 = ex2(fmaf(__uint_as_float(sr[k]), p.scale_log2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(sr[k + 1]), p.scale_log2, -m_use));
          sum += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS + 32 * half, pk);
      }
      l += sum;
      if (b > 0 && __any_sync(0xffffffffu, need)) {
        // O holds blocks < b (PV of block b-1 completed before S of block b
        // was committed); bring it to the new reference max
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * j, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(tO + 32 * j, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[t]);
    }
    if (ok) ok = warp_wait(&bars->o_done, 0, bars, p.status);
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow =
          p.out + ((int64_t)(off + tok) * p.Hq + (int64_t)kvh * p.g + row % p.g) * D;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * j, o);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * j);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
      }
    }
  } else if (warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    const int ptid = tid - kSoftmaxWarps * 32;
    const int ci = ptid & 7;
    const int rbase = ptid >> 3;  // rows rbase + kRowStep * i
    // Q tiles
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int row = rbase + kRowStep * i;
        const int tok = q0 + t * p.tpt + row / p.g;
        const bool valid = row < p.rows_used && tok < e;
        const __nv_bfloat16* src =
            p.q + ((int64_t)(off + (valid ? tok : 0)) * p.Hq + (int64_t)kvh * p.g + row % p.g) * D + ci * 8;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          cp_async_16(sQ_a + t * C::kTileBytes + c * C::kChunkBytes + sw128(row, ci),
                      valid ? src + c * 64 : p.q, valid ? 16u : 0u);
      }
    }
    cp_async_commit();
    int issued = 1, published = 0;
    auto publish_oldest = [&]() {
      fence_proxy_async_smem();
      if (published == 0) mbar_arrive(&bars->q_full);
      else mbar_arrive(&bars->kv_full[(published - 1) % C::kStages]);
      ++published;
    };
    const int32_t* rtt = p.req_to_token + (int64_t)p.req_pool_idx[r] * p.rtt_stride;
    int32_t slot_cur[kRowsPerThread], slot_next[kRowsPerThread];
    auto load_slots = [&](int b, int32_t (&dst)[kRowsPerThread]) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int j = b * BN + rbase + kRowStep * i;
        dst[i] = (b < nb_pre && j < pfx) ? rtt[j] : -1;
      }
    };
    if (nb_pre > 0) load_slots(0, slot_next);
    bool ok = true;
    for (int tile = 0; tile < 2 * nb && ok; ++tile) {
      const int b = tile >> 1, is_v = tile & 1;
      const int stage = tile % C::kStages, round = tile / C::kStages;
      if (round > 0) {
        ok = warp_wait(&bars->kv_empty[stage], (round - 1) & 1, bars, p.status);
        if (!ok) break;
      }
      if (!is_v) {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) slot_cur[i] = slot_next[i];
      }
      const uint32_t dst0 = sKV_a + stage * C::kTileBytes;
      if (b < nb_pre) {
        const __nv_bfloat16* pool = is_v ? p.pool_v : p.pool_k;
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int row = rbase + kRowStep * i;
          const bool valid = slot_cur[i] >= 0;
          const __nv_bfloat16* src =
              pool + ((int64_t)(valid ? slot_cur[i] : 0) * p.Hkv + kvh) * D + ci * 8;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            cp_async_16(dst0 + c * C::kChunkBytes + sw128(row, ci), src + c * 64, valid ? 16u : 0u);
        }
      } else {
        const __nv_bfloat16* base = is_v ? p.v_new : p.k_new;
        const int j0 = (b - nb_pre) * BN;
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int row = rbase + kRowStep * i;
          const int j = j0 + row;
          const bool valid = j < q_end;
          const __nv_bfloat16* src =
              base + ((int64_t)(off + (valid ? j : 0)) * p.Hkv + kvh) * D + ci * 8;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            cp_async_16(dst0 + c * C::kChunkBytes + sw128(row, ci), src + c * 64, valid ? 16u : 0u);
        }
      }
      cp_async_commit();
      ++issued;
      if (is_v && b + 1 < nb_pre) load_slots(b + 1, slot_next);
      if (issued - published > kLag) {
        cp_async_wait<kLag>();
        publish_oldest();
      }
    }
    cp_async_wait_all();
    if (ok)
      while (published < issued) publish_oldest();
  } else if (lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = make_idesc_bf16(BM, BN, false);
    constexpr uint32_t idO = make_idesc_bf16(BM, D, true);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return mbar_wait_bounded(bar, parity, &bars->abort, p.status);
    };
    auto issue_s = [&](int t, int stage) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
        const uint64_t a = make_sw128_desc(sQ_a + t * C::kTileBytes + o, 16, 1024);
        const uint64_t bd = make_sw128_desc(sKV_a + stage * C::kTileBytes + o, 16, 1024);
        umma_ss(tmem + col_s(t), a, bd, idS, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t bd =
            make_sw128_desc(sKV_a + stage * C::kTileBytes + kk * 16 * 128, C::kChunkBytes, 1024);
        umma_ts(tmem + col_o(t), tmem + col_s(t) + kk * 8, bd, idO, (acc || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = wait(&bars->q_full, 0);
    if (ok) tc_fence_after();
    for (int b = 0; b < nb && ok; ++b) {
      const int kt = 2 * b, ks = kt % C::kStages;
      if (!(ok = wait(&bars->kv_full[ks], (kt / C::kStages) & 1))) break;
      tc_fence_after();
      int vt = 0, vs = 0;
      if (b > 0) {
        vt = 2 * b - 1;
        vs = vt % C::kStages;
        if (!(ok = wait(&bars->p_ready[0], (b - 1) & 1))) break;
        if (!(ok = wait(&bars->kv_full[vs], (vt / C::kStages) & 1))) break;
        tc_fence_after();
        issue_pv(0, vs, b > 1);
      }
      issue_s(0, ks);
      umma_commit(&bars->s_full[0]);
      if (b > 0) {
        if (!(ok = wait(&bars->p_ready[1], (b - 1) & 1))) break;
        tc_fence_after();
        issue_pv(1, vs, b > 1);
        umma_commit(&bars->kv_empty[vs]);
      }
      issue_s(1, ks);
      umma_commit(&bars->s_full[1]);
      umma_commit(&bars->kv_empty[ks]);
    }
    if (ok) {
      const int vt = 2 * nb - 1, vs = vt % C::kStages;
      ok = wait(&bars->p_ready[0], (nb - 1) & 1) && wait(&bars->kv_full[vs], (vt / C::kStages) & 1);
      if (ok) {
        tc_fence_after();
        issue_pv(0, vs, nb > 1);
        ok = wait(&bars->p_ready[1], (nb - 1) & 1);
        if (ok) {
          tc_fence_after();
          issue_pv(1, vs, nb > 1);
          umma_commit(&bars->kv_empty[vs]);
          umma_commit(&bars->o_done);
        }
      }
    }
    if (!ok) {
      // let every MMA issued so far finish before TMEM is released
      umma_commit(&bars->drain);
      mbar_wait_bounded(&bars->drain, 0, &bars->abort, nullptr, 2000000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
sgl_status run(const Params& prm, int32_t batch, int32_t max_extend, cudaStream_t stream) {
  using C = Cfg<D>;
  auto kern = extend_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return SGL_ERR_CUDA;
  const int per_cta = 2 * prm.tpt;
  const unsigned gx = (unsigned)((max_extend + per_cta - 1) / per_cta);
  dim3 grid(gx, (unsigned)prm.Hkv, (unsigned)batch);
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? SGL_OK : SGL_ERR_CUDA;
}

}  // namespace

size_t extend_workspace_bytes() { return 256; }

sgl_status launch_extend(const ExtendArgs& a, cudaStream_t stream) {
  if (a.batch == 0 || a.total_extend == 0 || a.max_extend == 0) return SGL_OK;
  const int g = a.num_q_heads / a.num_kv_heads;
  if (g < 1 || g > BM) return SGL_ERR_UNSUPPORTED;
  if (a.batch > 65535 || a.num_kv_heads > 65535) return SGL_ERR_UNSUPPORTED;
  Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.pool_k = static_cast<const __nv_bfloat16*>(a.pool_k);
  prm.pool_v = static_cast<const __nv_bfloat16*>(a.pool_v);
  prm.req_to_token = a.req_to_token;
  prm.rtt_stride = a.rtt_stride;
  prm.req_pool_idx = a.req_pool_idx;
  prm.prefix_lens = a.prefix_lens;
  prm.extend_lens = a.extend_lens;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.Hq = a.num_q_heads;
  prm.Hkv = a.num_kv_heads;
  prm.g = g;
  prm.tpt = BM / g;
  prm.rows_used = prm.tpt * g;
  prm.scale_log2 = a.sm_scale * 1.4426950408889634f;
  prm.status = static_cast<int*>(a.workspace);
  if (a.head_dim == 128) return run<128>(prm, a.batch, a.max_extend, stream);
  if (a.head_dim == 64) return run<64>(prm, a.batch, a.max_extend, stream);
  return SGL_ERR_UNSUPPORTED;
}

}  // namespace sgl
