// Paged decode attention: one query per request over all of its slots.
//
// "Inside SGLang", Step 3 (Prefill and decode have different shapes): a
// decode step reads the key and value of every earlier token, so it is bound
// by memory bandwidth; (Paged KV and the kernels that read it): the kernel
// reads the request's slot indices from req_to_token and gathers its keys and
// values from wherever they sit in the pool.
//
// Schedule (split-KV):
//   1. plan    -- one block lists the work items (request, split): a
//                 request's keys are cut into ceil(seq_len / 1024) runs of
//                 near-equal length;
//   2. split   -- a persistent grid (x: one wave of CTAs taking items from a
//                 per-KV-head counter; y: KV head) runs
//                 each item: the slot indices go to shared memory, K and V
//                 rows of the KV head are gathered by 16-byte cp.async into a
//                 ring of tiles (CUDA-core path: 6 stages of 16 bf16 / 32 e4m3
//                 keys; tensor-core path: 4 stages of 32 / 64), and
//                 the query heads of the group share every loaded row.  Each
//                 warp takes a quarter of a tile: with one or two query heads
//                 per KV head on CUDA cores (LPT = 8 or 16 lanes own one key,
//                 each lane a slice of the head dim, every lane group an fp32
//                 online-softmax state), with four or more on tensor cores
//                 (warp-level MMAs whose rows are the query heads).  The
//                 warps' states are merged at the end of the item.  Requests
//                 with one split write the output directly; others write
//                 their partial state;
//   3. combine -- one warp per (request, query head) merges the partial
//                 states of multi-split requests (max-rescaled sums).
// Cascade decode (shared prefixes read once per group) runs the same three
// kernels with a group pass before the split: the plan kernel derives each
// request's shared length and group count from the groups, the split kernel
// covers only the private tail [shared_len, seq_len), and the combine merges
// the group states (written by the tensor-core group kernel) with the tail's.
// Scores are kept in the log2 domain (scale * log2(e) folded into q) and the
// running max is only moved when a score exceeds it by more than 2^8, which
// keeps every exponentiated weight <= 256 in fp32 and makes rescaling rare.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace sgl {
namespace dec {
namespace {

// keys per work item: kChunk, or kChunkLong when max_seq_len reaches
// kLongSeq (chunked-mix decode 6,705 -> 6,782 GB/s, tree decode unchanged;
// 2,048-key items cost Llama-7B-like decode 28%: too few items); kItemMax is
// the most any item holds (the slot run's shared-memory buffer)
constexpr int kChunk = 1024;
constexpr int kChunkLong = 1536;
constexpr int kItemMax = 1536;
// keys per work item when a unit covers kWarps KV heads (span gathers).
// Shorter items add partial states for the combine, longer ones leave too
// few units to even out the last round.  e4m3 tokens/s against 512-key items
// (measured): 384 keys -2% to -8%; 768 keys +4.4% on the tree cascade (its
// ~520-key private tails become one item each), +1.1% on the chunked mix
// (contexts up to 32 K), -2.7% on Llama-7B-like (64 requests of 0.5-4 K)
// and -0.9% on the tree's plain decode.  A call takes 768-key items for a
// cascade's tails or when max_seq_len reaches kLongSeq, else 512.
constexpr int kSpanChunk = 512;
constexpr int kSpanChunkLong = 768;
constexpr int kLongSeq = 16384;
static_assert(kChunkLong <= kItemMax && kSpanChunkLong <= kItemMax, "slot run buffer");
constexpr int kTileBf16 = 32;  // tensor-core path: bf16 keys per pipeline stage (twice as many e4m3)
constexpr int kStages = 4;     // tensor-core path: ring depth
// the CUDA-core path (measured best there: a deeper ring of smaller tiles)
constexpr int kTileBf16Fma = 16;
constexpr int kStagesFma = 6;
// resident split CTAs an SM on the tensor-core path (4 stages at 3 CTAs
// measured against 3 stages at 4: within 0.5% on most workloads)
constexpr int kMmaMinBlocks = 3;
// the e4m3 path with both products on the tensor core (E4m3MmaState): 3
// stages at 4 CTAs an SM (128 registers); measured against 4 stages at 3
// CTAs (160 registers): chunked-mix e4m3 decode 5,322 against 5,235 GB/s
// (and at one head per KV head 4,550 against 3,210)
constexpr int kStagesE4m3 = 3;
constexpr int kE4m3MinBlocks = 4;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Ws {
  int32_t* item_start;  // [B+1]
  int2* items;          // [max_items]
  int32_t* n_items;     // [1]
  int32_t* next_item;   // [Hkv] work counters (zeroed by the plan kernel)
  int2* req_info;       // [B] (shared_len, number of groups); cascade only, else null
  float2* part_ml;      // [max_items + B*max_depth, Hkv, G]  (max in log2 units, sum)
  float* part_acc;      // [max_items + B*max_depth, Hkv, G, D]
};

// The groups of a cascade decode (all null / 0 for plain decode).
struct Groups {
  const int32_t* start;
  const int32_t* len;
  const int32_t* depth;
  const int32_t* member_off;
  const int32_t* members;
  int32_t n_groups, max_depth;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline int64_t max_items_for(int32_t batch, int32_t max_seq_len, int32_t chunk) {
  return (int64_t)batch * ((max_seq_len + chunk - 1) / chunk);
}

// partial-state entries: the split items, then (cascade) B x max_depth group states
inline size_t ws_layout(int32_t batch, int64_t max_items, int32_t Hkv, int32_t G, int32_t D,
                        int32_t max_depth, bool cascade, void* base, Ws* ws) {
  const int64_t n_part = max_items + (cascade ? (int64_t)batch * max_depth : 0);
  size_t off = 0;
  size_t o_start = off;
  off = align256(off + sizeof(int32_t) * (size_t)(batch + 1));
  size_t o_items = off;
  off = align256(off + sizeof(int2) * (size_t)max_items);
  size_t o_n = off;
  off = align256(off + sizeof(int32_t));
  size_t o_next = off;
  off = align256(off + sizeof(int32_t) * (size_t)Hkv);
  size_t o_info = off;
  if (cascade) off = align256(off + sizeof(int2) * (size_t)batch);
  size_t o_ml = off;
  off = align256(off + sizeof(float2) * (size_t)n_part * Hkv * G);
  size_t o_acc = off;
  off = align256(off + sizeof(float) * (size_t)n_part * Hkv * G * D);
  if (ws && base) {
    char* b = static_cast<char*>(base);
    ws->item_start = reinterpret_cast<int32_t*>(b + o_start);
    ws->items = reinterpret_cast<int2*>(b + o_items);
    ws->n_items = reinterpret_cast<int32_t*>(b + o_n);
    ws->next_item = reinterpret_cast<int32_t*>(b + o_next);
    ws->req_info = cascade ? reinterpret_cast<int2*>(b + o_info) : nullptr;
    ws->part_ml = reinterpret_cast<float2*>(b + o_ml);
    ws->part_acc = reinterpret_cast<float*>(b + o_acc);
  }
  return off;
}

struct Params {
  const __nv_bfloat16* q;
  const uint8_t* pool_k;  // [S, Hkv, D] rows of bf16 or e4m3 values
  const uint8_t* pool_v;
  const int32_t* req_to_token;
  int64_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  __nv_bfloat16* out;
  // Hkv: KV heads as the kernels see them.  A group of more than 16 query
  // heads per KV head runs as kv_split "virtual" KV heads of Hq / Hkv query
  // heads each (virtual head v reads pool head v / kv_split; query heads,
  // outputs and partial states keep the same flat order); Hkv_pool is the
  // pool's own KV head count (the row stride of a slot).
  int32_t batch, Hq, Hkv;
  int32_t kv_split, Hkv_pool;
  int32_t chunk;  // keys per work item (chunk_for)
  float scale_log2;  // softmax scale * log2(e) * K scale (1 for a bf16 pool)
  float v_scale;     // V scale of an e4m3 pool (1 for bf16), applied to the output
  Ws ws;
  int64_t group_base;  // first partial entry of the group states (= max_items)
  int32_t max_depth;   // group states per request (cascade), else 0
};

// ---------------------------------------------------------------- plan

// (counters: kMixCounters words a mixed-batch launch takes work from, zeroed
// here when given)
constexpr int kMixCounters = 3;
__global__ void __launch_bounds__(1024) decode_plan_kernel(const int32_t* __restrict__ seq_lens,
                                                           int32_t batch, int64_t max_items, int32_t chunk,
                                                           int32_t Hkv, Ws ws, Groups gr,
                                                           int32_t* counters = nullptr) {
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dep_launch();  // the split kernel may start; it waits for this plan
  for (int h = tid; h < Hkv; h += blockDim.x) ws.next_item[h] = 0;
  if (counters != nullptr && tid < kMixCounters) counters[tid] = 0;
  if (ws.req_info != nullptr) {
    // cascade: every membership raises its request's shared length to the
    // group's end and its group count to the group's depth + 1
    for (int r = tid; r < batch; r += blockDim.x) ws.req_info[r] = make_int2(0, 0);
    __syncthreads();
    for (int j = warp; j < gr.n_groups; j += blockDim.x >> 5) {
      const int32_t a = gr.member_off[j], b = gr.member_off[j + 1];
      const int32_t end = gr.start[j] + gr.len[j], cnt = gr.depth[j] + 1;
      for (int32_t k = a + lane; k < b; k += 32) {
        const int32_t r = gr.members[k];
        if (r >= 0 && r < batch) {
          atomicMax(&ws.req_info[r].x, end);
          atomicMax(&ws.req_info[r].y, min(cnt, gr.max_depth));
        }
      }
    }
    __syncthreads();
  }
  // keys of request r handled by split items: the private tail [shared_len, seq_len)
  auto tail_len = [&](int r) {
    const int32_t sh = ws.req_info != nullptr ? __ldcg(&ws.req_info[r].x) : 0;
    return max(seq_lens[r] - sh, 0);
  };
  const int per = (batch + blockDim.x - 1) / blockDim.x;
  const int r0 = min(batch, tid * per), r1 = min(batch, r0 + per);
  int32_t local = 0;
  for (int r = r0; r < r1; ++r) local += (tail_len(r) + chunk - 1) / chunk;
  // block-wide exclusive scan of `local`
  int32_t inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int32_t t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  int32_t base = inc - local + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int r = r0; r < r1; ++r) {
    ws.item_start[r] = base;
    const int32_t ns = (tail_len(r) + chunk - 1) / chunk;
    for (int32_t s = 0; s < ns; ++s)
      if (base + s < max_items) ws.items[base + s] = make_int2(r, s);
    base += ns;
  }
  if (tid == blockDim.x - 1) {
    ws.item_start[batch] = base;
    *ws.n_items = (int32_t)min((int64_t)base, max_items);
  }
}

// ---------------------------------------------------------------- split

// LPT lanes own one key; each lane holds D/LPT elements of the head dim, in
// chunks of at most 16 bytes of the stored row (8 bf16 or 16 e4m3 values);
// the LPT lanes' chunks are contiguous, so a warp's loads are coalesced.
// LPT = 8 for small head groups, 16 when G*D is large (keeps the per-lane
// query and accumulator registers bounded).  KV is the pool's element type:
// __nv_bfloat16, or uint8_t holding e4m3 codes.
template <int D, int LPT, typename KV>
struct Lane {
  static constexpr int kBytes = (int)sizeof(KV);
  static constexpr int kRowBytes = D * kBytes;
  static constexpr int kRowVecs = kRowBytes / 16;  // 16-byte vectors per row
  static constexpr int kElems = D / LPT;           // elements per lane
  static constexpr int kChunkElems = (16 / kBytes) < kElems ? (16 / kBytes) : kElems;
  static constexpr int kChunks = kElems / kChunkElems;
  static constexpr int kGroups = 32 / LPT;         // keys per warp instruction
  // element offset of chunk c of lane li
  static __device__ __forceinline__ int elem(int c, int li) {
    return c * (kChunkElems * LPT) + li * kChunkElems;
  }
};

// n stored values of type KV at p -> n floats (e4m3 codes are exact in float)
template <typename KV, int N>
SGL_DEV void load_row_chunk(const uint8_t* p, float* f) {
  if constexpr (sizeof(KV) == 2) {
    static_assert(N == 8, "one 16-byte vector of bf16");
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(p), f);
  } else {
    static_assert(N == 8 || N == 16, "8 or 16 e4m3 codes");
    uint32_t w[N / 4];
    if constexpr (N == 16) {
      const uint4 v = *reinterpret_cast<const uint4*>(p);
      w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x, w[1] = v.y;
    }
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
            (__nv_fp8x2_storage_t)(w[i] >> (16 * h)), __NV_E4M3);
        const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&r));
        f[4 * i + 2 * h] = x.x;
        f[4 * i + 2 * h + 1] = x.y;
      }
    }
  }
}

template <int D, int G, int LPT>
__host__ __device__ constexpr int min_blocks() { return 2 * G * D / LPT <= 64 ? 3 : 2; }

// Which (pool type, group size) take the tensor-core path (measured best):
// three or more query heads per KV head, or two or more on an e4m3 pool.
// With one or two bf16 query heads per KV head the 16-row MMAs carry 14-15
// empty rows and the CUDA-core path is faster (7-8%); from four heads on the
// MMAs remove most of the per-key instructions (tree decode 23% faster at
// G = 4); above 8 heads the MMA rows 8..15 carry heads too.  On e4m3 pools
// with 2 or 4 heads both products take the codes as they are (E4m3MmaState);
// with other group sizes MmaState widens them by bit placement on the integer pipe (code
// * 2^-8 as f16, the 2^8 folded back into the scores and the published sums;
// the hardware e4m3x2 -> f16x2 conversion measured the same).
template <typename KV, int G>
__host__ __device__ constexpr bool use_mma() {
  return G >= 3 || (sizeof(KV) == 1 && G >= 2);
}
// e4m3 pools with 2 or 4 query heads per KV head: both products on e4m3
// MMAs, no widening (E4m3MmaState).  With one head the CUDA-core path stays
// (Llama-7B-like e4m3 decode 4,710 against 4,570 GB/s on this one: the MMAs
// cost the same per key at any group size, the CUDA-core work halves)
template <typename KV, int G>
__host__ __device__ constexpr bool use_e4m3_mma() {
  return sizeof(KV) == 1 && (G == 2 || G == 4);
}

// Per-warp attention state of the CUDA-core path: LPT lanes own one key, each
// lane a slice of the head dim; every lane group keeps an fp32 online-softmax
// state (max, sum, weighted V sum) for each of the G query heads.
template <int D, int G, int LPT, typename KV, int kTile>
struct FmaState {
  using L = Lane<D, LPT, KV>;
  static constexpr int kSwizzle = 0;  // plain ring rows
  static constexpr int EL = L::kElems, CE = L::kChunkElems;
  float qf[G][EL];
  float m[G], l[G], acc[G][EL];
  int grp, li, warp;

  SGL_DEV void init(int lane, int w) {
    grp = lane / LPT;
    li = lane % LPT;
    warp = w;
  }
  // this lane's slice of the G query heads, pre-scaled into log2 units
  SGL_DEV void load_q(const __nv_bfloat16* qb, float scale_log2) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
        for (int u = 0; u < CE; u += 8) {
          uint4 raw = *reinterpret_cast<const uint4*>(qb + h * D + L::elem(c, li) + u);
          bf16x8_to_f32(raw, &qf[h][c * CE + u]);
#pragma unroll
          for (int e = 0; e < 8; ++e) qf[h][c * CE + u + e] *= scale_log2;
        }
  }
  SGL_DEV void reset() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < EL; ++e) acc[h][e] = 0.f;
    }
  }
  // the stage's keys key0 .. key0 + kTile (those < n are valid)
  SGL_DEV void stage(const uint8_t* ks, const uint8_t* vs, int key0, int n, float) {
#pragma unroll
    for (int sub = 0; sub < kTile / (L::kGroups * kWarps); ++sub) {
      const int tok = warp * (kTile / kWarps) + sub * L::kGroups + grp;
      const bool valid = key0 + tok < n;
      float kf[EL];
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        load_row_chunk<KV, CE>(ks + tok * L::kRowBytes + L::kBytes * L::elem(c, li), &kf[c * CE]);
      // q.k and p.v on the packed fp32 pipe (two lanes of FMA per instruction)
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < EL; e += 2)
          a = ffma2(make_float2(qf[h][e], qf[h][e + 1]), make_float2(kf[e], kf[e + 1]), a);
        s[h] = a.x + a.y;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = 1; o < LPT; o <<= 1) s[h] += __shfl_xor_sync(0xffffffffu, s[h], o);
        if (!valid) s[h] = -INFINITY;
      }
      bool need = false;
#pragma unroll
      for (int h = 0; h < G; ++h) need |= s[h] > m[h] + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (s[h] > m[h] + kRescaleThreshold) {
            const float a = ex2(m[h] - s[h]);
            m[h] = s[h];
            l[h] *= a;
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[h][e] *= a;
          }
        }
      }
      float vf[EL];
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        load_row_chunk<KV, CE>(vs + tok * L::kRowBytes + L::kBytes * L::elem(c, li), &vf[c * CE]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pw = valid ? ex2(s[h] - m[h]) : 0.f;
        l[h] += pw;
#pragma unroll
        for (int e = 0; e < EL; e += 2) {
          const float2 a = ffma2(make_float2(pw, pw), make_float2(vf[e], vf[e + 1]),
                                 make_float2(acc[h][e], acc[h][e + 1]));
          acc[h][e] = a.x;
          acc[h][e + 1] = a.y;
        }
      }
    }
  }
  // merge the warp's lane groups and write its state to the CTA scratch
  SGL_DEV void publish(float* red_acc, float* red_m, float* red_l) {
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float mn = fmaxf(m[h], mo);
        const float fa = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
        const float fb = mo == -INFINITY ? 0.f : ex2(mo - mn);
        l[h] = l[h] * fa + lo * fb;
#pragma unroll
        for (int e = 0; e < EL; ++e) {
          const float ao = __shfl_xor_sync(0xffffffffu, acc[h][e], off);
          acc[h][e] = acc[h][e] * fa + ao * fb;
        }
        m[h] = mn;
      }
    }
    if (grp == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
          for (int e = 0; e < CE; ++e)
            red_acc[(warp * G + h) * D + L::elem(c, li) + e] = acc[h][c * CE + e];
        if (li == 0) {
          red_m[warp * G + h] = m[h];
          red_l[warp * G + h] = l[h];
        }
      }
    }
  }
};

// Per-warp attention state of the tensor-core path: the G query heads are the
// rows of warp-level MMAs (m16n8k16 / m16n8k8, rows G..15 zero), lane (g, t)
// = (lane / 4, lane % 4).  q.k contracts over the head dim in an order both
// operands share (lane t holds dims [t*D/4, (t+1)*D/4) of its row, four per
// k-step), so each lane's K row slice is one run of 16-byte loads; p.v
// permutes the output columns so that lane g's V loads are contiguous (n-col
// g of 8-column block j of 32-column block sb is dim 32*sb + 4*g + j; lane
// (g, t) ends up holding dims 32*sb + 8*t .. +7 of head g).  bf16 pools use
// bf16 operands; e4m3 pools convert codes to f16 operands two at a time.
// Accumulation and the online softmax stay fp32; P is rounded to the operand
// type before the p.v product.
template <int D, int G, typename KV, int kTile>
struct MmaState {
  static constexpr int kSwizzle = 0;  // plain ring rows
  static constexpr int kBytes = (int)sizeof(KV);
  static constexpr int kRowBytes = D * kBytes;
  static constexpr int KS = D / 16;          // k-steps of q.k
  static constexpr int SB = D / 32;          // 32-column blocks of p.v
  static constexpr int KW = kTile / kWarps;  // keys of a warp per stage: 8 bf16, 16 e4m3
  static constexpr int DL = D / 4;           // head-dim values of one lane in q.k
  static constexpr bool kTwoRows = G > 8;    // rows 8..15 carry heads too
  static constexpr int NR = kTwoRows ? 2 : 1;  // rows of a lane: g (and g + 8)
  static_assert(G <= 16, "at most 16 query heads per KV head");
  static_assert(KW == (kBytes == 2 ? 8 : 16), "stage shape");
  uint32_t qa[KS][2 * NR];  // per k-step: row g lo, row g hi (, row g+8 lo, row g+8 hi)
  float o[SB][4][4];        // c0, c1: row g; c2, c3: row g + 8
  float m[NR], l[NR];
  int g, t, warp;

  SGL_DEV void init(int lane, int w) {
    g = lane >> 2;
    t = lane & 3;
    warp = w;
  }
  SGL_DEV void load_q(const __nv_bfloat16* qb, float) {
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      const int row = g + 8 * rr;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) qa[ks][2 * rr] = qa[ks][2 * rr + 1] = 0u;
      if (row < G) {
        const uint4* src = reinterpret_cast<const uint4*>(qb + row * D + DL * t);
#pragma unroll
        for (int v = 0; v < DL / 8; ++v) {
          const uint4 w = src[v];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t x = ws[i];
            if constexpr (kBytes == 1)
              x = pack_f16x2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
            qa[(4 * v + i) / 2][2 * rr + (4 * v + i) % 2] = x;
          }
        }
      }
    }
  }
  SGL_DEV void reset() {
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      m[rr] = -INFINITY;
      l[rr] = 0.f;
    }
#pragma unroll
    for (int b = 0; b < SB; ++b)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[b][j][c] = 0.f;
  }
  SGL_DEV void qk(float (&d4)[4], int ks_, uint32_t b0, uint32_t b1) {
    uint32_t a1 = 0u, a3 = 0u;  // rows g + 8
    if constexpr (kTwoRows) {
      a1 = qa[ks_][2];
      a3 = qa[ks_][3];
    }
    if constexpr (kBytes == 2) {
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d4[0]), "+f"(d4[1]), "+f"(d4[2]), "+f"(d4[3])
          : "r"(qa[ks_][0]), "r"(a1), "r"(qa[ks_][1]), "r"(a3), "r"(b0), "r"(b1));
    } else {
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d4[0]), "+f"(d4[1]), "+f"(d4[2]), "+f"(d4[3])
          : "r"(qa[ks_][0]), "r"(a1), "r"(qa[ks_][1]), "r"(a3), "r"(b0), "r"(b1));
    }
  }
  // widened e4m3 operands hold code * 2^-8
  static constexpr float kWiden = kBytes == 1 ? 256.f : 1.f;
  SGL_DEV static void widen4(uint32_t w, uint32_t& lo, uint32_t& hi) { e4m3x4_to_f16x2_scaled(w, lo, hi); }
  SGL_DEV void stage(const uint8_t* ks, const uint8_t* vs, int key0, int n, float scale_log2_in) {
    // widened K codes hold code * 2^-8
    const float scale_log2 = scale_log2_in * kWiden;
    // ---- S = q.k for this warp's KW keys, 8 at a time; sv[nb][row set][c]
    float sv[KW / 8][NR][2];
#pragma unroll
    for (int nb = 0; nb < KW / 8; ++nb) {
      const uint8_t* row = ks + (warp * KW + nb * 8 + g) * kRowBytes + DL * t * kBytes;
      float d4[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kBytes == 2) {
#pragma unroll
        for (int v = 0; v < DL / 8; ++v) {  // 8 bf16 = two k-steps
          const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * v);
          qk(d4, 2 * v, w.x, w.y);
          qk(d4, 2 * v + 1, w.z, w.w);
        }
      } else {
#pragma unroll
        for (int v = 0; v < DL / 16; ++v) {  // 16 codes = four k-steps
          const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * v);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t lo, hi;
            widen4(ws[i], lo, hi);
            qk(d4, 4 * v + i, lo, hi);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < NR; ++rr)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          sv[nb][rr][c] =
              key0 + warp * KW + nb * 8 + 2 * t + c < n ? d4[2 * rr + c] * scale_log2 : -INFINITY;
    }
    // ---- online softmax of row g (and g + 8); the 4 lanes of a row agree on m
    float pv[KW / 8][NR][2];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float mx = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < KW / 8; ++nb) mx = fmax3(mx, sv[nb][rr][0], sv[nb][rr][1]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m[rr] + kRescaleThreshold) {
        const float a = m[rr] == -INFINITY ? 0.f : ex2(m[rr] - mx);
        m[rr] = mx;
        l[rr] *= a;
#pragma unroll
        for (int b = 0; b < SB; ++b)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[b][j][2 * rr] *= a;
            o[b][j][2 * rr + 1] *= a;
          }
      }
#pragma unroll
      for (int nb = 0; nb < KW / 8; ++nb)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          pv[nb][rr][c] = sv[nb][rr][c] == -INFINITY ? 0.f : ex2(sv[nb][rr][c] - m[rr]);
          l[rr] += pv[nb][rr][c];
        }
    }
    // ---- O += P V
    const uint8_t* r0 = vs + (warp * KW + 2 * t) * kRowBytes;  // key 2t of this warp's keys
    if constexpr (kBytes == 2) {
      const uint32_t a0 = pack_bf16x2(pv[0][0][0], pv[0][0][1]);
      const uint32_t a1 = kTwoRows ? pack_bf16x2(pv[0][NR - 1][0], pv[0][NR - 1][1]) : 0u;
#pragma unroll
      for (int b = 0; b < SB; ++b) {
        const uint2 x = *reinterpret_cast<const uint2*>(r0 + 2 * (32 * b + 4 * g));
        const uint2 y = *reinterpret_cast<const uint2*>(r0 + kRowBytes + 2 * (32 * b + 4 * g));
        const uint32_t bj[4] = {__byte_perm(x.x, y.x, 0x5410), __byte_perm(x.x, y.x, 0x7632),
                                __byte_perm(x.y, y.y, 0x5410), __byte_perm(x.y, y.y, 0x7632)};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm volatile(
              "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
              "{%0,%1,%2,%3};"
              : "+f"(o[b][j][0]), "+f"(o[b][j][1]), "+f"(o[b][j][2]), "+f"(o[b][j][3])
              : "r"(a0), "r"(a1), "r"(bj[j]));
      }
    } else {
      const uint32_t a0 = pack_f16x2(pv[0][0][0], pv[0][0][1]), a2 = pack_f16x2(pv[1][0][0], pv[1][0][1]);
      const uint32_t a1 = kTwoRows ? pack_f16x2(pv[0][NR - 1][0], pv[0][NR - 1][1]) : 0u;
      const uint32_t a3 = kTwoRows ? pack_f16x2(pv[1][NR - 1][0], pv[1][NR - 1][1]) : 0u;
#pragma unroll
      for (int b = 0; b < SB; ++b) {
        const int col = 32 * b + 4 * g;
        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(r0 + col);
        const uint32_t x1 = *reinterpret_cast<const uint32_t*>(r0 + kRowBytes + col);
        const uint32_t y0 = *reinterpret_cast<const uint32_t*>(r0 + 8 * kRowBytes + col);
        const uint32_t y1 = *reinterpret_cast<const uint32_t*>(r0 + 9 * kRowBytes + col);
        const uint32_t xa = __byte_perm(x0, x1, 0x5140), xb = __byte_perm(x0, x1, 0x7362);
        const uint32_t ya = __byte_perm(y0, y1, 0x5140), yb = __byte_perm(y0, y1, 0x7362);
        uint32_t b0[4], b1[4];
        widen4(xa, b0[0], b0[1]);
        widen4(xb, b0[2], b0[3]);
        widen4(ya, b1[0], b1[1]);
        widen4(yb, b1[2], b1[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
              "{%8,%9}, {%0,%1,%2,%3};"
              : "+f"(o[b][j][0]), "+f"(o[b][j][1]), "+f"(o[b][j][2]), "+f"(o[b][j][3])
              : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0[j]), "r"(b1[j]));
      }
    }
  }
  SGL_DEV void publish(float* red_acc, float* red_m, float* red_l) {
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) {
      float ls = l[rr];
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      const int row = g + 8 * rr;
      if (row < G) {
        float* dst = red_acc + (warp * G + row) * D + 8 * t;
#pragma unroll
        for (int b = 0; b < SB; ++b)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dst[32 * b + j] = o[b][j][2 * rr] * kWiden;  // back to code units
            dst[32 * b + 4 + j] = o[b][j][2 * rr + 1] * kWiden;
          }
        if (t == 0) {
          red_m[warp * G + row] = m[rr];
          red_l[warp * G + row] = ls;
        }
      }
    }
  }
};

// Per-warp attention state over an e4m3 pool with 2 or 4 query heads per KV
// head: both products on e4m3 tensor-core MMAs (m16n8k32, fp32
// accumulation), no code widened.
//
// q.k: the A rows hold each head's query as three e4m3 terms (hi + mid + lo:
// ~12 significant bits, the head scaled by a power of two into e4m3's
// range), term j of head h in row j * G + h, so one MMA computes all three;
// the B columns are keys.  Lane g's rows are g and g + 8: with G = 2 head g's
// terms are the rows g, g + 2, g + 4 of lanes 8 and 16 on (two shuffles add
// them); with G = 4 they are rows g and g + 8 of the lane itself and row
// g + 4 of the lane 16 on.  The warp's 16 keys of a stage go
// to the columns of two MMAs so that, after the sums, lane (h, t) holds head
// h's scores of keys 4t .. 4t + 3: the keys its p.v operand needs.
//
// p.v: A = V^T (16 head dims x 32 keys) straight from the ring by the
// transposing 8-bit ldmatrix, keys 16..31 zero (a warp has 16 keys a stage);
// B = P as two e4m3 terms of x = 2^8 p, hi = e4m3(x) and lo = e4m3(x - hi)
// (~8 significant bits, as a bf16 P), column j * G + h holding term j of head
// h.  The reference max is exact (moved whenever a block raises it), so p <=
// 1 and x <= 256 fits e4m3; x and the row sums carry 2^8 until the state is
// published.
//
// The ring rows are XOR-swizzled by 16-byte chunk (chunk c of row r at c ^ (r
// & kSwizzle)), so the 8-row phases of both products' loads hit distinct banks.
template <int D, int G, int kTile>
struct E4m3MmaState {
  static constexpr int kRowBytes = D;
  static constexpr int kSwizzle = D / 16 - 1;  // 16-byte chunks a row, less one
  static constexpr int KW = kTile / kWarps;    // keys of a warp per stage
  static constexpr int DL = D / 4;             // head dims of one lane in q.k
  static constexpr int KS8 = D / 32;           // k-steps of q.k
  static constexpr int DB = D / 16;            // 16-dim blocks of p.v
  static_assert(KW == 16, "16 keys a warp per stage");
  static_assert(G == 2 || G == 4, "group sizes of this path");
  uint32_t q8[KS8][4];  // a0..a3 of k-step ks (rows g, g + 8; k = 4t.., 16 + 4t..)
  float qmul;           // 2^-e of head g (rows g < G)
  float c[DB][4];       // p.v: rows (dims) 16 b + g, 16 b + 8 + g; columns 2t, 2t + 1
  float m, l;           // head g's reference max and row sum (lanes g < G)
  int g, t, warp;

  SGL_DEV void init(int lane, int w) {
    g = lane >> 2;
    t = lane & 3;
    warp = w;
  }
  SGL_DEV void load_q(const __nv_bfloat16* qb, float) { load_q_terms(qb); }
  // Row g = j * G + h (j < 3): term j of head h, over this lane's dims
  // DL * t .. DL * t + DL - 1 (the same dims its K loads cover), in k-step
  // order: k-step ks holds dims 8 ks .. 8 ks + 7 of the slice, four a word.
  // The head's scale 2^e puts its largest |q| in [128, 256) (the four lanes of
  // a row hold its four slices); hi = e4m3(q 2^e), mid = e4m3(q 2^e - hi),
  // lo = e4m3(q 2^e - hi - mid), each difference exact in fp32.
  SGL_DEV void load_q_terms(const __nv_bfloat16* qb) {
    // rows g and g + 8 belong to the same head (G divides 8) as terms
    // g / G and (g + 8) / G
    const int h = g % G, term0 = g / G, term1 = (g + 8) / G;
    const bool live = g < 3 * G;
    float x[DL];
    float amax = 0.f;
#pragma unroll
    for (int v = 0; v < DL / 8; ++v) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (live) raw = *reinterpret_cast<const uint4*>(qb + h * D + DL * t + 8 * v);
      bf16x8_to_f32(raw, &x[8 * v]);
    }
#pragma unroll
    for (int i = 0; i < DL; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;
    if (amax > 0.f) e = min(126, max(-126, 7 - (((__float_as_int(amax) >> 23) & 0xff) - 127)));
    const float sc = __int_as_float((e + 127) << 23);
    qmul = __int_as_float((127 - e) << 23);
#pragma unroll
    for (int ks = 0; ks < KS8; ++ks)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t w0 = 0u, w1 = 0u;
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
          const int d = 8 * ks + 4 * hf + i;
          float2 v = make_float2(x[d] * sc, x[d + 1] * sc);
          uint32_t c0 = 0u, c1 = 0u;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const __nv_fp8x2_storage_t cj = __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);
            if (j == term0) c0 = (uint32_t)cj;
            if (j == term1) c1 = (uint32_t)cj;
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(cj, __NV_E4M3);
            const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            v = make_float2(v.x - back.x, v.y - back.y);
          }
          w0 |= c0 << (8 * i);
          w1 |= c1 << (8 * i);
        }
        q8[ks][2 * hf] = live ? w0 : 0u;                      // row g
        q8[ks][2 * hf + 1] = live && term1 < 3 ? w1 : 0u;     // row g + 8
      }
  }
  SGL_DEV void qk8(float (&d4)[4], int ks_, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d4[0]), "+f"(d4[1]), "+f"(d4[2]), "+f"(d4[3])
        : "r"(q8[ks_][0]), "r"(q8[ks_][1]), "r"(q8[ks_][2]), "r"(q8[ks_][3]), "r"(b0), "r"(b1));
  }
  SGL_DEV void reset() {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int b = 0; b < DB; ++b)
#pragma unroll
      for (int k = 0; k < 4; ++k) c[b][k] = 0.f;
  }
  SGL_DEV void stage(const uint8_t* ks, const uint8_t* vs, int key0, int n, float scale_log2_in) {
    const float scale_log2 = scale_log2_in * qmul;  // the scores carry the head's 2^e
    // ---- S: column g of MMA nb is key 4 (g / 2) + 2 nb + g % 2 of the warp's
    // 16, so lane (h, t) ends with head h's scores of keys 4t + 2 nb + cc
    float s[2][2];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const int r = warp * KW + 4 * (g >> 1) + 2 * nb + (g & 1);
      const uint8_t* row = ks + r * kRowBytes;
      float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int v = 0; v < DL / 16; ++v) {  // 16 codes = two k-steps
        const int chunk = ((DL / 16) * t + v) ^ (r & kSwizzle);
        const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * chunk);
        qk8(d4, 2 * v, w.x, w.y);
        qk8(d4, 2 * v + 1, w.z, w.w);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        if constexpr (G == 4)
          d4[cc] += __shfl_down_sync(0xffffffffu, d4[cc], 16) + d4[cc + 2];
        else
          d4[cc] += __shfl_down_sync(0xffffffffu, d4[cc], 4 * G) + __shfl_down_sync(0xffffffffu, d4[cc], 8 * G);
        s[nb][cc] = key0 + warp * KW + 4 * t + 2 * nb + cc < n ? d4[cc] * scale_log2 : -INFINITY;
      }
    }
    // ---- online softmax of head g over its 16 keys (lanes g < G); the
    // reference moves whenever the block max is above it
    float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (__any_sync(0xffffffffu, g < G && mx > m)) {
      const float mn = fmaxf(m, mx);
      const float a = m == -INFINITY ? 0.f : ex2(m - mn);
      m = mn;
      l *= a;
      // accumulator columns 2t, 2t + 1 belong to heads 2t % G, (2t + 1) % G
      const float a0 = __shfl_sync(0xffffffffu, a, 4 * ((2 * t) % G));
      const float a1 = __shfl_sync(0xffffffffu, a, 4 * ((2 * t + 1) % G));
#pragma unroll
      for (int b = 0; b < DB; ++b) {
        c[b][0] *= a0;
        c[b][2] *= a0;
        c[b][1] *= a1;
        c[b][3] *= a1;
      }
    }
    // ---- P terms of keys 4t .. 4t + 3, one byte a key
    uint32_t hi = 0u, lo = 0u;
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      const float x0 = s[nb][0] == -INFINITY ? 0.f : ex2(s[nb][0] - m + 8.f);
      const float x1 = s[nb][1] == -INFINITY ? 0.f : ex2(s[nb][1] - m + 8.f);
      l += x0 + x1;
      const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
      const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_fp8x2_storage_t l2 =
          __nv_cvt_float2_to_fp8x2(make_float2(x0 - back.x, x1 - back.y), __NV_SATFINITE, __NV_E4M3);
      hi |= (uint32_t)h2 << (16 * nb);
      lo |= (uint32_t)l2 << (16 * nb);
    }
    // column g: hi of head g (g < G, this lane), lo of head g - G (G <= g <
    // 2G, the lane 4G before), else zero
    const uint32_t lo_up = __shfl_up_sync(0xffffffffu, lo, 4 * G);
    const uint32_t b0 = g < G ? hi : (g < 2 * G ? lo_up : 0u);
    // ---- O^T += V^T P: ldmatrix rows are the warp's 16 keys (lanes 16..31
    // repeat the addresses of lanes 0..15)
    const int kr = warp * KW + ((4 * g + t) & 15);
    const uint8_t* vrow = vs + kr * kRowBytes;
#pragma unroll
    for (int b = 0; b < DB; ++b) {
      uint32_t a0, a1;
      asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0,%1}, [%2];"
                   : "=r"(a0), "=r"(a1)
                   : "r"(smem_u32(vrow + 16 * (b ^ (kr & kSwizzle)))));
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[b][0]), "+f"(c[b][1]), "+f"(c[b][2]), "+f"(c[b][3])
          : "r"(a0), "r"(a1), "r"(0u), "r"(0u), "r"(b0), "r"(0u));
    }
  }
  SGL_DEV void publish(float* red_acc, float* red_m, float* red_l) {
    constexpr float kUnscale = 1.f / 256.f;  // x and the sums carry 2^8
    float ls = l + __shfl_xor_sync(0xffffffffu, l, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    if (g < G && t == 0) {
      red_m[warp * G + g] = m;
      red_l[warp * G + g] = ls * kUnscale;
    }
    // head h's hi and lo sit in columns h and G + h: the next lane (G = 2)
    // or the lane two on (G = 4)
#pragma unroll
    for (int b = 0; b < DB; ++b) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = c[b][k] + __shfl_down_sync(0xffffffffu, c[b][k], G / 2);
      if (t < G / 2) {
        const int h0 = 2 * t;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          red_acc[(warp * G + h0 + (k & 1)) * D + 16 * b + 8 * (k >> 1) + g] = v[k] * kUnscale;
      }
    }
  }
};

template <int D, int G, int LPT, typename KV>
__host__ __device__ constexpr int split_min_blocks() {
  return use_e4m3_mma<KV, G>() ? kE4m3MinBlocks : use_mma<KV, G>() ? kMmaMinBlocks : min_blocks<D, G, LPT>();
}

// Ring shape of the split kernel: the tensor-core path takes 32 bf16 keys per
// stage (8 per warp), the CUDA-core path its own tile and depth.  A stage
// holds the same bytes for either pool type (twice as many e4m3 keys).
template <typename KV, int G>
struct SplitRing {
  static constexpr bool kMma = use_mma<KV, G>();
  static constexpr int kTileB = kMma ? kTileBf16 : kTileBf16Fma;  // bf16 keys per stage
  static constexpr int kDepth = use_e4m3_mma<KV, G>() ? kStagesE4m3 : kMma ? kStages : kStagesFma;
  static constexpr int kTile = kTileB * 2 / (int)sizeof(KV);            // keys per stage
  template <int D>
  static constexpr size_t bytes() { return (size_t)kDepth * 2 * kTileB * D * 2; }
};

// Split-KV work units run by one group of kWarps warps (kThreads threads):
// gtid is the thread's index in the group, sync() the group's barrier,
// next() (called by gtid 0) the group's next unit, n_units the end of the
// units and head_of(u) / item_of(u) the (KV head, work item) of unit u;
// smem holds the group's ring and slot run, s_item two words of the group's
// shared memory.  The split kernel runs one group a CTA over one KV head's
// items; the mixed batch kernel runs five groups a CTA over (item, KV head)
// units.
// kDepth: ring stages (0: the split kernel's).
// kSpans: head_of(u) is the first of kWarps adjacent KV heads (a multiple of
// kWarps; the pool holds them side by side in every slot) and warp w takes
// head head_of(u) + w: a stage holds kTile / kWarps keys of each of those
// heads, gathered as one contiguous span of kWarps rows a slot and laid out
// in shared memory head by head, so warp w finds its head's keys where a
// per-head stage keeps warp w's slice of the keys, and every warp's state is
// the whole item's for its head (no merge across warps).
template <int D, int G, int LPT, typename KV, int kDepth = 0, bool kSpans = false, class Sync, class Next,
          class HeadOf, class ItemOf>
SGL_DEV void split_units(const Params& p, uint8_t* smem, int32_t* s_item, int gtid, int32_t n_units, Sync sync,
                         Next next, HeadOf head_of, ItemOf item_of) {
  using L = Lane<D, LPT, KV>;
  using Ring = SplitRing<KV, G>;
  constexpr int kTile = Ring::kTile;  // keys per pipeline stage
  constexpr int kStages = kDepth > 0 ? kDepth : Ring::kDepth;
  constexpr int kTileBytes = kTile * L::kRowBytes;         // one K or V tile
  constexpr int kStageBytes = 2 * kTileBytes;              // K then V
  constexpr int KW = kTile / kWarps;                       // keys of a warp's slice of a stage
  constexpr int kStageKeys = kSpans ? KW : kTile;          // an item's keys a stage covers
  using State = std::conditional_t<
      use_e4m3_mma<KV, G>(), E4m3MmaState<D, G, kTile>,
      std::conditional_t<use_mma<KV, G>(), MmaState<D, G, KV, kTile>, FmaState<D, G, LPT, KV, kTile>>>;
  int32_t* s_slots = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes);
  float* s_red = reinterpret_cast<float*>(smem);           // reuses the ring after an item

  const int tid = gtid, lane = tid & 31, warp = tid >> 5;
  const uint32_t ring = smem_u32(smem);
  State st;
  st.init(lane, warp);
  // units are taken dynamically; the next index is fetched while the
  // current unit runs
  if (tid == 0) s_item[0] = next();
  sync();
  int buf = 0;

  for (int32_t unit = s_item[0]; unit < n_units; unit = s_item[buf]) {
    int32_t nxt = 0;
    if (tid == 0) nxt = next();
    const int kvh0 = head_of(unit);                // the unit's (first) KV head
    const int kvh = kSpans ? kvh0 + warp : kvh0;    // this warp's
    const int32_t item = item_of(unit);
    const int2 it = p.ws.items[item];
    const int r = it.x;
    // the request's keys past its shared groups (all of them in plain decode)
    // are cut into ceil(n / chunk) near-equal items
    const int2 info = p.ws.req_info != nullptr ? p.ws.req_info[r] : make_int2(0, 0);
    const int32_t tail = max(p.seq_lens[r] - info.x, 0);
    const int32_t ns = (tail + p.chunk - 1) / p.chunk;
    const int32_t base = tail / ns, rem = tail % ns;
    const int32_t t0 = info.x + it.y * base + min(it.y, rem);
    const int32_t n = base + (it.y < rem ? 1 : 0);
    const int32_t* rtt = p.req_to_token + (int64_t)p.req_pool_idx[r] * p.rtt_stride + t0;
    for (int i = tid; i < n; i += kThreads) s_slots[i] = rtt[i];
    st.load_q(p.q + ((int64_t)r * p.Hq + (int64_t)kvh * G) * D, p.scale_log2);
    sync();  // slots visible; previous item's reduction scratch free

    const int n_tiles = (n + kStageKeys - 1) / kStageKeys;
    const uint8_t* kbase = p.pool_k + (int64_t)(kvh0 / p.kv_split) * L::kRowBytes;
    const uint8_t* vbase = p.pool_v + (int64_t)(kvh0 / p.kv_split) * L::kRowBytes;
    auto issue = [&](int tile, int stage) {
      const uint32_t st_a = ring + stage * kStageBytes;
      if constexpr (kSpans) {
        // consecutive threads copy consecutive 16-byte pieces of a slot's span
        // of kWarps rows; piece (w, vec) of key j lands in row w * KW + j
        constexpr int kSpanVecs = kWarps * L::kRowVecs;
        constexpr int kKeysPerPass = kThreads / kSpanVecs;
        static_assert(kThreads % kSpanVecs == 0 && KW % kKeysPerPass == 0, "span copy shape");
        const int w = (tid % kSpanVecs) / L::kRowVecs, vec = tid % L::kRowVecs;
#pragma unroll
        for (int pass = 0; pass < KW / kKeysPerPass; ++pass) {
          const int key = pass * kKeysPerPass + tid / kSpanVecs;
          const int32_t j = tile * KW + key;
          const bool ok = j < n;
          const int64_t row = (ok ? (int64_t)s_slots[j] * p.Hkv_pool : 0) + w;
          const int tok = w * KW + key;
          const uint32_t d = st_a + tok * L::kRowBytes + (vec ^ (tok & State::kSwizzle)) * 16;
          cp_async_16(d, kbase + row * L::kRowBytes + vec * 16, ok ? 16u : 0u);
          cp_async_16(d + kTileBytes, vbase + row * L::kRowBytes + vec * 16, ok ? 16u : 0u);
        }
      } else {
        constexpr int kRowsPerPass = kThreads / L::kRowVecs;
        const int vec = tid % L::kRowVecs;
#pragma unroll
        for (int pass = 0; pass < kTile / kRowsPerPass; ++pass) {
          const int tok = pass * kRowsPerPass + tid / L::kRowVecs;
          const int32_t j = tile * kTile + tok;
          const bool ok = j < n;
          const int64_t row = ok ? (int64_t)s_slots[j] * p.Hkv_pool : 0;
          const uint32_t d = st_a + tok * L::kRowBytes + (vec ^ (tok & State::kSwizzle)) * 16;
          cp_async_16(d, kbase + row * L::kRowBytes + vec * 16, ok ? 16u : 0u);
          cp_async_16(d + kTileBytes, vbase + row * L::kRowBytes + vec * 16, ok ? 16u : 0u);
        }
      }
    };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < n_tiles) issue(s, s);
      cp_async_commit();
    }
    st.reset();
    for (int k = 0; k < n_tiles; ++k) {
      cp_async_wait<kStages - 2>();
      sync();
      if (k + kStages - 1 < n_tiles) issue(k + kStages - 1, (k + kStages - 1) % kStages);
      cp_async_commit();
      const uint8_t* ks = smem + (k % kStages) * kStageBytes;
      // a state masks key key0 + warp * KW + i of its slice
      st.stage(ks, ks + kTileBytes, kSpans ? (k - warp) * KW : k * kTile, n, p.scale_log2);
    }
    cp_async_wait_all();

    sync();  // every warp is done with the ring; reuse it for the reduction
    // s_red layout: [warp][G][D] acc, then [warp][G] m, then [warp][G] l
    float* red_acc = s_red;
    float* red_m = s_red + kWarps * G * D;
    float* red_l = red_m + kWarps * G;
    st.publish(red_acc, red_m, red_l);
    sync();
    const bool single = ns == 1 && info.y == 0;
    // (head, query head, dim) outputs of the unit: kWarps heads with spans
    constexpr int kHeads = kSpans ? kWarps : 1;
    for (int idx = tid; idx < kHeads * G * D; idx += kThreads) {
      const int wh = idx / (G * D), h = (idx / D) % G, d = idx % D;
      float M, Ls, A;
      if constexpr (kSpans) {
        // warp wh's state covers the whole item for head kvh0 + wh
        M = red_m[wh * G + h];
        Ls = red_l[wh * G + h];
        A = red_acc[(wh * G + h) * D + d];
      } else {
        M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * G + h]);
        Ls = 0.f;
        A = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float mw = red_m[w * G + h];
          const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
          Ls += red_l[w * G + h] * f;
          A += red_acc[(w * G + h) * D + d] * f;
        }
      }
      const int head = kvh0 + wh;
      if (single) {
        p.out[((int64_t)r * p.Hq + (int64_t)head * G + h) * D + d] = __float2bfloat16_rn(A * (p.v_scale / Ls));
      } else {
        const int64_t slot = ((int64_t)item * p.Hkv + head) * G + h;
        p.ws.part_acc[slot * D + d] = A;
        if (d == 0) p.ws.part_ml[slot] = make_float2(M, Ls);
      }
    }
    if (tid == 0) s_item[buf ^ 1] = nxt;
    buf ^= 1;
    sync();  // scratch, slots and the next item index
  }
}


// kSpans = false: one group a CTA over the items of KV head blockIdx.y,
// taken from that head's counter.  kSpans = true: over the items of the
// kWarps adjacent KV heads kWarps * blockIdx.y.., one warp a head, each slot's
// rows of those heads gathered as one span (counter blockIdx.y).
template <int D, int G, int LPT, typename KV, bool kSpans>
__global__ void __launch_bounds__(kThreads, (split_min_blocks<D, G, LPT, KV>()))
decode_split_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t s_item[2];
  const int y = blockIdx.y;
  // launched dependent on the plan: a cascade's group pass (launched
  // dependent on this kernel) may take the SMs this grid leaves; then wait
  // for the plan's items and counters
  grid_dep_launch();
  grid_dep_wait();
  split_units<D, G, LPT, KV, 0, kSpans>(
      p, smem, s_item, threadIdx.x, *p.ws.n_items, [] { __syncthreads(); },
      [&] { return atomicAdd(&p.ws.next_item[y], 1); }, [&](int32_t) { return kSpans ? kWarps * y : y; },
      [](int32_t u) { return u; });
}

// ---------------------------------------------------------------- combine

template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(Params p) {
  grid_dep_wait();  // launched dependent on the split kernel (or the group pass)
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (gw >= (int64_t)p.batch * p.Hq) return;
  const int r = (int)(gw / p.Hq), h = (int)(gw % p.Hq);
  const int32_t s0 = p.ws.item_start[r];
  const int32_t n_split = p.ws.item_start[r + 1] - s0;
  const int32_t n_grp = p.ws.req_info != nullptr ? p.ws.req_info[r].y : 0;
  if (n_grp == 0 && n_split <= 1) return;     // a single split wrote the output
  if (s0 + n_split > *p.ws.n_items) return;   // lengths above max_seq_len
  const int32_t ns = n_grp + n_split;
  const int G = p.Hq / p.Hkv;
  const int kvh = h / G, hh = h % G;
  // states in key order: the groups by depth, then the tail's splits
  auto slot_of = [&](int32_t s) {
    const int64_t e = s < n_grp ? p.group_base + (int64_t)r * p.max_depth + s : (int64_t)(s0 + s - n_grp);
    return (e * p.Hkv + kvh) * G + hh;
  };
  float M = -INFINITY;
  for (int32_t s = lane; s < ns; s += 32) M = fmaxf(M, p.ws.part_ml[slot_of(s)].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float Ls = 0.f;
  for (int32_t s = 0; s < ns; ++s) {
    const int64_t sl = slot_of(s);
    const float2 ml = p.ws.part_ml[sl];
    const float f = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
    Ls += ml.y * f;
    const float* a = p.ws.part_acc + sl * D;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(f, a[lane + 32 * e], acc[e]);
  }
  const float inv = p.v_scale / Ls;
  __nv_bfloat16* o = p.out + ((int64_t)r * p.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < E; ++e) o[lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
}

// Split factor for groups of more than 16 query heads per KV head: the
// smallest s dividing G with G / s <= 16 (1 for G <= 16).
inline int32_t kv_split_for(int32_t G) {
  if (G <= 16) return 1;
  for (int32_t s = 2; s <= G; ++s)
    if (G % s == 0 && G / s <= 16) return s;
  return G;
}

// A decode over an e4m3 pool gathers a slot's rows of kWarps adjacent KV
// heads as one span (512 bytes at head dim 128 instead of four 128-byte rows:
// random 128-byte rows read at 4.6-4.8 TB/s on this part, 512-byte spans at
// 6.9) when its (kernel) KV heads come in whole groups of kWarps, each its
// own pool head; its items then hold kSpanChunk or kSpanChunkLong keys.  Measured with e4m3
// pools: chunked mix +3.9%, Llama-7B-like +4.0%, tree cascade +3.2% (tokens
// a second).  bf16 pools keep one KV head a unit (256-byte rows already read
// at 6.6-6.8 TB/s; spans measured +1.0% on the chunked mix, -0.6% on
// Llama-7B-like and -6% on the tree cascade, whose short private tails leave
// too few span units).  spans_possible: the bound the workspace is sized for.
inline bool spans_possible(int32_t Hkv, int32_t kv_split) { return kv_split == 1 && Hkv % kWarps == 0; }
inline bool spans_for(int32_t Hkv, int32_t kv_split, bool kv_fp8) { return kv_fp8 && spans_possible(Hkv, kv_split); }
inline int32_t chunk_for(bool spans) { return spans ? kSpanChunk : kChunk; }  // the shortest a call takes
inline int32_t chunk_for(bool spans, bool cascade, int32_t max_seq_len) {
  if (!spans) return max_seq_len >= kLongSeq ? kChunkLong : kChunk;
  return cascade || max_seq_len >= kLongSeq ? kSpanChunkLong : kSpanChunk;
}

// The kernel parameters of a decode call: the workspace layout and, for a
// cascade decode, the group pass's arguments.
struct DecodePlan {
  int G;              // query heads of a (virtual) KV head
  int64_t max_items;  // work items the workspace holds
  Groups gr;
  GroupArgs ga;
  bool groups;        // a cascade with groups to attend
};
inline sgl_status make_decode_params(const DecodeArgs& a, Params* prm, DecodePlan* pl) {
  const int G_pool = a.num_q_heads / a.num_kv_heads;
  const int split = kv_split_for(G_pool);
  const int G = G_pool / split;                 // query heads of a (virtual) KV head
  const int Hkv = a.num_kv_heads * split;       // KV heads as the kernels see them
  const int64_t max_items = max_items_for(a.batch, a.max_seq_len, chunk_for(spans_possible(Hkv, split)));
  prm->chunk = chunk_for(spans_for(Hkv, split, a.kv_fp8), a.cascade, a.max_seq_len);
  prm->q = static_cast<const __nv_bfloat16*>(a.q);
  prm->pool_k = static_cast<const uint8_t*>(a.pool_k);
  prm->pool_v = static_cast<const uint8_t*>(a.pool_v);
  prm->req_to_token = a.req_to_token;
  prm->rtt_stride = a.rtt_stride;
  prm->req_pool_idx = a.req_pool_idx;
  prm->seq_lens = a.seq_lens;
  prm->out = static_cast<__nv_bfloat16*>(a.out);
  prm->batch = a.batch;
  prm->Hq = a.num_q_heads;
  prm->Hkv = Hkv;
  prm->kv_split = split;
  prm->Hkv_pool = a.num_kv_heads;
  // the K scale of an e4m3 pool folds into the query, the V scale into the output
  prm->scale_log2 = a.sm_scale * 1.4426950408889634f * (a.kv_fp8 ? a.k_scale : 1.f);
  prm->v_scale = a.kv_fp8 ? a.v_scale : 1.f;
  // cascade: word 0 of the workspace is the group pass's status; the decode
  // scratch follows the status bytes
  const size_t head = a.cascade ? kCascadeStatusBytes : 0;
  const int32_t max_depth = a.cascade ? a.max_depth : 0;
  char* base = static_cast<char*>(a.workspace);
  if (base == nullptr) return SGL_ERR_WORKSPACE;
  const size_t need = head + ws_layout(a.batch, max_items, Hkv, G, a.head_dim, max_depth,
                                       a.cascade, base + head, &prm->ws);
  if (a.workspace_bytes < need) return SGL_ERR_WORKSPACE;
  prm->group_base = max_items;
  prm->max_depth = max_depth;
  Groups gr = {};
  GroupArgs ga = {};
  const bool groups = a.cascade && a.n_groups > 0;
  if (groups) {
    gr = Groups{a.group_start, a.group_len, a.group_depth, a.group_member_off, a.group_members,
                a.n_groups, max_depth};
    ga.q = a.q;
    ga.pool_k = a.pool_k;
    ga.pool_v = a.pool_v;
    ga.req_to_token = a.req_to_token;
    ga.rtt_stride = a.rtt_stride;
    ga.req_pool_idx = a.req_pool_idx;
    ga.group_start = a.group_start;
    ga.group_len = a.group_len;
    ga.group_depth = a.group_depth;
    ga.member_off = a.group_member_off;
    ga.members = a.group_members;
    ga.batch = a.batch;
    ga.n_groups = a.n_groups;
    ga.max_members = a.max_group_members;
    ga.max_depth = max_depth;
    ga.part_ml = prm->ws.part_ml;
    ga.part_acc = prm->ws.part_acc;
    ga.part_base = max_items;
    ga.status = reinterpret_cast<int*>(base);
    ga.num_q_heads = a.num_q_heads;
    ga.num_kv_heads = a.num_kv_heads;
    ga.head_dim = a.head_dim;
    ga.sm_scale = a.sm_scale;
    ga.kv_fp8 = a.kv_fp8;
    ga.k_scale = a.k_scale;
  }
  pl->G = G;
  pl->max_items = max_items;
  pl->gr = gr;
  pl->ga = ga;
  pl->groups = groups;
  return SGL_OK;
}

}  // namespace
}  // namespace dec
}  // namespace sgl
