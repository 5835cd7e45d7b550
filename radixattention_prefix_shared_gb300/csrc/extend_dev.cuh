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
// Warp roles (19 warps):
//   warps 0-15 softmax: Q tile t = (w/4)%2, TMEM lane quarter w%4, key-column
//              half w/8 -- two warps share the rows of a lane quarter, each
//              taking 64 of the block's 128 keys.  Idle until the first S,
//              they also issue the Q tiles' copies; at the end they write the
//              output through shared memory (each thread deposits its row,
//              each warp stores whole rows with consecutive lanes)
//   warps 16-17 producers: 16-byte cp.async gathers of K and V rows into
//              the 128-byte-swizzled shared-memory layout the tensor core
//              reads; each thread's arrival on the stage's mbarrier fires in
//              hardware when its copies land (cp.async.mbarrier.arrive), so a
//              producer never waits for its own copies; the MMA thread orders
//              the landed data for the tensor core with a proxy fence
//   warp 18    TMEM allocation and the single thread that issues tcgen05.mma
// TMEM (512 columns): S0 | S1 | O0 | O1.  S_t = Q_t K^T lands in TMEM as
// fp32; the softmax warps read it, write P = exp2(S*scale*log2e - m) as
// bf16 over the first half of S_t's columns, and O_t += P V is issued with A
// read from TMEM.  The two Q tiles ping-pong: while softmax works on one
// tile the tensor core computes the other.  The reference max used for the
// exponentials lags the running max lazily: a block is accepted while its
// row sum stays <= 2^32 (every weight then fits fp32 and bf16 with full
// relative precision); otherwise the block max becomes the reference and O
// is rescaled in TMEM, so most blocks need neither a max pass nor a
// correction pass.
//
// e4m3 pool: every key and value -- the suffix too, stored before the call --
// is gathered through req_to_token as codes.  Three producer warps stage the
// codes with cp.async and widen them to f16 into the swizzled ring with
// integer ops, and the softmax runs as 8 warps that own whole rows (one
// thread a row, all 128 keys of a block; no pair vote), so each producer
// shares its sub-partition with two softmax warps instead of four: the code's seven magnitude bits placed
// at f16 bit 7 (sign at bit 15) read as exactly code * 2^-8, subnormal codes
// included, so both MMAs run on f16 operands (the query is widened from bf16,
// P is packed as f16 with the lazy bound lowered to 2^15) and the 2^8 and the
// pool's scales fold into the softmax scale and the output.
//
// Every wait on an mbarrier is bounded (2 s); on a timeout the kernel raises
// an abort flag, records a status word in the workspace, drains its own
// in-flight copies and MMAs, frees TMEM and returns.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace sgl {
namespace ext {
namespace {

constexpr int BM = 128;  // rows per Q tile
constexpr int BN = 128;  // keys per KV block
// e4m3 codes widened by bit placement hold code * 2^-8
constexpr float kFp8Operand = 256.0f;
// Q tiles a cascade-group CTA holds over a bf16 pool
constexpr int kGroupTilesBf16 = 1;
// e4m3 pools: f16 ring stages at D = 128 (twice as many at D = 64), raw code
// staging slots, and code rows a producer thread loads before it stores
// (measured: 2 staging slots -15%, half-tile staging units with 4 stages -9%)
constexpr int kFp8Stages = 3;
constexpr int kFp8RawSlots = 3;
constexpr int kFp8Batch = 5;

// registers a thread the kernels that split their registers are built with
// (16 warps over an e4m3 pool: 128; 20 warps over a bf16 pool: 96), checked
// before their launch: the split below is exact for it
template <bool kFp8>
constexpr int split_launch_regs() { return kFp8 ? 128 : 96; }

// warp roles: softmax warps, producer warps, the MMA warp, with registers
// moved between warpgroups by setmaxnreg after the setup barrier (not in the
// mixed batch kernel's persistent tiles, whose warps run decode work too).
// e4m3: seven producer warps (each K/V code is copied and widened by the
// producers, the kernel's limit), 16 warps launched at 128 registers a
// thread -- the two softmax warpgroups (whole rows) take 160, the producers'
// and the MMA warp's give up to 96 -- against three producers in 12 warps at
// 168 (extend 785 -> 1,062 TFLOP/s on the chunked mix, 803 -> 1,034 on the
// shared prompt).  bf16, two Q tiles: three producer warps, 20 warps
// launched at 96 -- the four softmax warpgroups take 104, the producers' and
// the MMA warp's give up to 64 -- against two producers in 19 warps at 96
// (1,221 -> 1,277 TFLOP/s on the chunked mix, 1,186 -> 1,236 on the shared
// prompt).  kTiles: Q tiles of 128 rows a CTA (2, ping-pong; 1 for the
// cascade group pass over bf16 pools, small enough for two CTAs an SM, no
// split)
template <bool kFp8, int kTiles = 2>
struct Roles {
  // softmax: on e4m3 pools 8 warps owning whole rows (one thread a row, all
  // 128 keys of a block); on bf16 pools 16 warps in pairs splitting each
  // row's keys (measured: whole rows equal on bf16 pools, +10% on e4m3 pools,
  // whose producers then share each sub-partition with two softmax warps
  // instead of four)
  static constexpr bool kFullRows = kFp8;
  static constexpr int kSoftmaxWarps = (kFullRows ? 4 : 8) * kTiles;
  static constexpr int kProducerWarps = kFp8 ? 7 : (kTiles == 2 ? 3 : 2);
  // register split (setmaxnreg.inc / .dec after the setup barrier), exact
  // for the launch's registers so the increase always finds what the
  // decrease releases: e4m3 8 x 32 x 160 + 8 x 32 x 96 = 512 x 128 (measured:
  // 168 / 88 -2%, 152 / 104 -1%, 144 / 112 -3%); bf16 16 x 32 x 104 +
  // 4 x 32 x 64 = 640 x 96
  static constexpr bool kSplitRegs = kFp8 || kTiles == 2;
  static constexpr int kSoftmaxRegs = kFp8 ? 160 : 104, kOtherRegs = kFp8 ? 96 : 64;
  static constexpr int kLaunchRegs = split_launch_regs<kFp8>();
  static constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;
  static constexpr int kThreads = (kMmaWarp + 1) * 32;
  static constexpr int kProducerThreads = kProducerWarps * 32;
  // a producer thread copies 16-byte chunk (ptid % 8) of the bf16 rows
  // ptid / 8 + kRowStep * i < 128, i < kRowsPerThread, of every 128-row tile
  static constexpr int kRowStep = kProducerThreads / 8;
  static constexpr int kRowsPerThread = (128 + kRowStep - 1) / kRowStep;
  // largest accepted block row sum: every weight must fit the P operand
  // (bf16: 2^32; f16: 2^15 < 65504)
  static constexpr float kAcceptSum = kFp8 ? 32768.0f : 4294967296.0f;
};
// TMEM columns: S_0 .. S_{kTiles-1}, then O_0 .. O_{kTiles-1}
template <int kTiles>
constexpr uint32_t tmem_cols() { return 256u * kTiles; }
SGL_DEV constexpr uint32_t col_s(int t) { return 128u * t; }
template <int kTiles>
SGL_DEV constexpr uint32_t col_o(int t) { return 128u * kTiles + 128u * t; }

template <int D, bool kFp8, int kTiles = 2>
struct Cfg {
  static constexpr int kChunks = D / 64;            // 128-byte column chunks per row
  static constexpr int kChunkBytes = 128 * 128;     // 128 rows x 128 bytes
  static constexpr int kTileBytes = 128 * D * 2;    // Q tile or one K / V block (16-bit)
  // K/V ring slots of 16-bit operands (4 keep the next block's K loading
  // while the current block's last MMAs still read the slot of the one
  // before: fewer put the widening of K on the tensor core's critical path)
  // (one Q tile: two stages, which keeps two CTAs on an SM)
  static constexpr int kStages = kTiles == 1 ? (D == 128 ? 2 : 4)
                                 : kFp8      ? (D == 128 ? kFp8Stages : 2 * kFp8Stages)
                                             : (D == 128 ? 4 : 8);
  static_assert(kTiles == 2 || !kFp8, "one Q tile only over bf16 pools");
  // e4m3: staging slots of raw codes ("units" of kUnitRows rows x D bytes,
  // unswizzled; one unit a tile)
  static constexpr int kUnitRows = 128;
  static constexpr int kUnits = 128 / kUnitRows;  // units per tile
  static constexpr int kRaw = kFp8 ? (D == 128 ? kFp8RawSlots : 4) : 0;
  static constexpr int kRawTileBytes = kUnitRows * D;
  static constexpr int kRawChunks = D / 16;  // 16-byte code chunks per row
  static constexpr int kRawRowStep = Roles<kFp8>::kProducerThreads / kRawChunks;
  static constexpr int kRawRows = (kUnitRows + kRawRowStep - 1) / kRawRowStep;  // rows a thread, per unit

  static_assert(Roles<kFp8>::kProducerThreads % 8 == 0 && Roles<kFp8>::kProducerThreads % kRawChunks == 0,
                "producer chunk columns");
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
  float xchg[2][2][128];  // [tile][column half][row]: block maxima, final row sums
};

// The kernel's dynamic shared memory, from its first 1024-byte boundary (the
// launch adds 1024 bytes of slack).
SGL_DEV uint8_t* smem_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

// The barriers, past the Q tiles, the ring and the raw code staging.
template <int D, bool kFp8, int kTiles>
SGL_DEV Bars* bars_of(uint8_t* smem) {
  using C = Cfg<D, kFp8, kTiles>;
  return reinterpret_cast<Bars*>(smem + (kTiles + C::kStages) * C::kTileBytes + C::kRaw * C::kRawTileBytes);
}

// Initialise every barrier a tile uses (one arrival each), so that a
// persistent CTA's first tile finds valid barriers to invalidate.
template <int kStagesUsed>
SGL_DEV void init_barriers_once(Bars* b) {
  mbar_init(&b->q_full, 1);
  for (int t = 0; t < 2; ++t) {
    mbar_init(&b->s_full[t], 1);
    mbar_init(&b->p_ready[t], 1);
  }
  mbar_init(&b->o_done, 1);
  mbar_init(&b->drain, 1);
  for (int s = 0; s < kStagesUsed; ++s) {
    mbar_init(&b->kv_full[s], 1);
    mbar_init(&b->kv_empty[s], 1);
  }
}

// Invalidate every barrier a tile uses (before they are initialised again).
template <int kStagesUsed>
SGL_DEV void invalidate_barriers(Bars* b) {
  mbar_inval(&b->q_full);
  for (int t = 0; t < 2; ++t) {
    mbar_inval(&b->s_full[t]);
    mbar_inval(&b->p_ready[t]);
  }
  mbar_inval(&b->o_done);
  mbar_inval(&b->drain);
  for (int s = 0; s < kStagesUsed; ++s) {
    mbar_inval(&b->kv_full[s]);
    mbar_inval(&b->kv_empty[s]);
  }
}

// dynamic shared memory: 1024 bytes of alignment slack, Q tiles, the K/V
// ring, the raw code staging (e4m3), barriers
template <int D, bool kFp8, int kTiles = 2>
constexpr int smem_bytes() {
  using C = Cfg<D, kFp8, kTiles>;
  return 1024 + (kTiles + C::kStages) * C::kTileBytes + C::kRaw * C::kRawTileBytes + (int)sizeof(Bars);
}
static_assert(smem_bytes<128, false>() <= 227 * 1024, "extend kernel shared memory");
static_assert(smem_bytes<64, false>() <= 227 * 1024, "extend kernel shared memory");
static_assert(smem_bytes<128, true>() <= 227 * 1024, "extend kernel shared memory");
static_assert(smem_bytes<64, true>() <= 227 * 1024, "extend kernel shared memory");
// one Q tile: two CTAs on an SM
static_assert(2 * smem_bytes<128, false, 1>() <= 228 * 1024 && 2 * smem_bytes<64, false, 1>() <= 228 * 1024,
              "two single-tile CTAs an SM");

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* pool_k;  // bf16 pool
  const __nv_bfloat16* pool_v;
  const uint8_t* pool_k8;  // e4m3 pool (codes)
  const uint8_t* pool_v8;
  const int32_t* req_to_token;
  int64_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* prefix_lens;
  const int32_t* extend_lens;
  __nv_bfloat16* out;
  int32_t Hq, Hkv, g, tpt, rows_used;
  float scale_log2;
  // multiplies the normalised output (extend) or the unnormalised P.V rows
  // (group mode); 1 on a bf16 pool
  float o_scale;
  int* status;
  uint64_t wait_ns;  // limit of every bounded wait on a stage barrier
  // group mode (cascade decode): group j covers positions
  // [group_start[j], group_start[j] + group_len[j]) of its members' rows and
  // its members are members[member_off[j] .. member_off[j+1]); the fp32 state
  // of member r, query head h goes to entry
  // ((part_base + r * max_depth + group_depth[j]) * Hkv + kvh) * g + h % g
  const int32_t* group_start;
  const int32_t* group_len;
  const int32_t* group_depth;
  const int32_t* member_off;
  const int32_t* members;
  float2* part_ml;  // (reference max in log2 units, row sum)
  float* part_acc;  // unnormalised P.V rows, D floats each
  int64_t part_base;
  int32_t max_depth;
  int32_t batch;  // member indices outside [0, batch) are skipped
};

// byte offset of 16-byte chunk `ci` (0..7) of row `row` inside one
// 128-row x 128-byte swizzled chunk
SGL_DEV uint32_t sw128(int row, int ci) { return row * 128 + ((ci ^ (row & 7)) << 4); }

// Warp-collective bounded wait: lane 0 polls, the verdict is broadcast.
SGL_DEV bool warp_wait(uint64_t* bar, uint32_t parity, Bars* bars, const Params& p) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, &bars->abort, p.status, p.wait_ns);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Epilogue staging.  Once o_done has fired no MMA reads the Q tiles or the
// K/V ring and no producer writes them, so that space holds the finished rows:
// row rr of tile t at byte (t * 128 + rr) * stride (rows padded by 16 bytes,
// so the 32 rows a warp deposits at once fall on different banks).  Each
// thread deposits its own row (the TMEM lane it read); the warp then writes
// its 32 rows out with consecutive lanes on consecutive 16-byte pieces of a
// row, instead of every lane storing into a different row.
template <int D>
constexpr int out_stride() { return 2 * D + 16; }  // bf16 output rows

// The warp's rows row0 .. row0+31 of a staged tile: kSeg bytes of each row at
// stage + rr * kStride go to dst(rr) (nullptr: the row holds no output).  The
// destination is recomputed per row from its index (measured faster than
// broadcasting each owner's pointer by shuffle).
template <int kSeg, int kStride, typename DstFn>
SGL_DEV void warp_store_rows(uint32_t stage, int row0, DstFn dst) {
  constexpr int kCpr = kSeg / 16;  // 16-byte pieces per row
  constexpr int kRpi = 32 / kCpr;  // rows per pass of the warp
  static_assert(kSeg % 16 == 0 && 32 % kCpr == 0, "row segment");
  const int lane = threadIdx.x & 31;
  __syncwarp();  // the warp's deposits are visible to the whole warp
#pragma unroll
  for (int i = 0; i < kCpr; ++i) {
    const int rr = row0 + i * kRpi + lane / kCpr, c = lane % kCpr;
    uint8_t* d = dst(rr);
    if (d != nullptr) *reinterpret_cast<uint4*>(d + 16 * c) = ld_shared_v4(stage + rr * kStride + 16 * c);
  }
}

// both tiles' staged rows fit in the Q tiles and the ring, below the
// barriers
template <int D, bool kFp8>
constexpr bool staging_fits() {
  using C = Cfg<D, kFp8>;
  return 256 * out_stride<D>() <= (2 + C::kStages) * C::kTileBytes;
}
static_assert(staging_fits<128, false>() && staging_fits<64, false>() && staging_fits<128, true>() &&
                  staging_fits<64, true>(),
              "epilogue staging");

// Whether the softmax warps, idle until the first S, load the Q tiles (so
// the producers start on K/V at once).  Always on bf16 pools; on e4m3 pools
// only in group mode (cascade groups: a few key blocks per CTA, so the
// prologue counts; measured there +5-7%, while on the chunked-prefill extend
// the producers' own Q load was 1.5% faster).
template <bool kFp8, bool kGroup>
constexpr bool q_by_softmax() { return !kFp8 || kGroup; }

// 16-byte cp.async copies of the two Q tiles into the swizzled K-major
// layout, spread over `nthreads` threads (ltid = index among them): chunk
// ltid % 8 of rows ltid / 8 + (nthreads / 8) * i.  Row m of tile t is token
// q0 + t * tpt + m / g, head m % g of the KV head's group; rows past the
// CTA's tokens are zero-filled.  Group mode gathers the members' decode
// queries.
template <int D, bool kGroup, int kTiles>
SGL_DEV void issue_q_copies(const Params& p, uint32_t sQ_a, int ltid, int nthreads, int kvh, int e, int mbeg,
                            int q0, int off) {
  using C = Cfg<D, false>;
  const int ci = ltid & 7, step = nthreads >> 3;
#pragma unroll
  for (int t = 0; t < kTiles; ++t) {
    for (int row = ltid >> 3; row < 128; row += step) {
      const int tok = q0 + t * p.tpt + row / p.g;
      bool valid = row < p.rows_used && tok < e;
      // the query row: suffix token off+tok, or member tok's decode query
      int64_t qrow = valid ? (kGroup ? (int64_t)p.members[mbeg + tok] : (int64_t)(off + tok)) : 0;
      if (kGroup && (qrow < 0 || qrow >= p.batch)) valid = false, qrow = 0;
      const __nv_bfloat16* src = p.q + (qrow * p.Hq + (int64_t)kvh * p.g + row % p.g) * D + ci * 8;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        cp_async_16(sQ_a + t * C::kTileBytes + c * C::kChunkBytes + sw128(row, ci),
                    valid ? src + c * 64 : p.q, valid ? 16u : 0u);
    }
  }
}

// e4m3 pools: the bf16 Q chunks this thread copied (the distribution of
// issue_q_copies) widened in place to f16, the operand type of both MMAs.
template <int D>
SGL_DEV void widen_q_in_place(uint32_t sQ_a, int ltid, int nthreads) {
  using C = Cfg<D, true>;
  const int ci = ltid & 7, step = nthreads >> 3;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    for (int row = ltid >> 3; row < 128; row += step) {
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const uint32_t a = sQ_a + t * C::kTileBytes + c * C::kChunkBytes + sw128(row, ci);
        const uint4 w = ld_shared_v4(a);
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          h[k] = pack_f16x2(__uint_as_float(x[k] << 16), __uint_as_float(x[k] & 0xFFFF0000u));
        st_shared_v4(a, h[0], h[1], h[2], h[3]);
      }
    }
  }
}

// The Q tiles loaded by the softmax warps (ltid = thread index among the
// nthreads of them), signalled on q_full: on a bf16 pool each thread's
// arrival fires when its copies land; on an e4m3 pool each thread waits for
// its own copies, widens them and orders them for the tensor core first.
template <int D, bool kGroup, bool kFp8, int kTiles>
SGL_DEV void load_q_tiles(const Params& p, uint32_t sQ_a, uint64_t* q_full, int ltid, int nthreads, int kvh,
                          int e, int mbeg, int q0, int off) {
  issue_q_copies<D, kGroup, kTiles>(p, sQ_a, ltid, nthreads, kvh, e, mbeg, q0, off);
  if constexpr (kFp8) {
    cp_async_wait_all();
    widen_q_in_place<D>(sQ_a, ltid, nthreads);
    fence_proxy_async_smem();
    mbar_arrive(q_full);
  } else {
    cp_async_mbar_arrive(q_full);
  }
}

// Producers on an e4m3 pool (Roles<true>::kProducerThreads threads, ptid =
// thread index among them; a thread's rows past the tile's end are
// skipped).  Q: the bf16 rows are copied like on a bf16 pool, then widened to
// f16 in place.  K/V: each key's D codes are copied with cp.async into an
// unswizzled staging slot of half a tile (one commit group per half, so a
// thread waits only for its own copies), widened by bit placement
// (code * 2^-8 as f16) and stored into the swizzled ring slot; the stores are
// ordered for the tensor core with a proxy fence before the arrival.  Prefix
// keys are positions 0..pfx-1 of the request's row, suffix keys positions
// pfx..pfx+q_end-1 (stored into the pool before the call).
template <int D, bool kGroup>
SGL_DEV void produce_fp8(const Params& p, uint32_t sQ_a, uint8_t* sKV, uint8_t* sRaw, Bars* bars,
                         int ptid, int r, int kvh, int e, int mbeg, int q0, int pfx, int q_end, int nb_pre, int nb,
                         int off) {
  const uint32_t sRaw_a = smem_u32(sRaw);
  using C = Cfg<D, true>;
  using R = Roles<true>;
  // ---- Q tiles (bf16 rows, 16-byte chunk ci of rows rbase + kRowStep * i),
  // unless the softmax warps load them
  const int ci = ptid & 7, rbase = ptid >> 3;
  if constexpr (!q_by_softmax<true, kGroup>()) {
#pragma unroll
  for (int t = 0; t < 2; ++t) {
#pragma unroll
    for (int i = 0; i < R::kRowsPerThread; ++i) {
      const int row = rbase + R::kRowStep * i;
      if (row >= 128) break;
      const int tok = q0 + t * p.tpt + row / p.g;
      bool valid = row < p.rows_used && tok < e;
      int64_t qrow = valid ? (kGroup ? (int64_t)p.members[mbeg + tok] : (int64_t)(off + tok)) : 0;
      if (kGroup && (qrow < 0 || qrow >= p.batch)) valid = false, qrow = 0;
      const __nv_bfloat16* src = p.q + (qrow * p.Hq + (int64_t)kvh * p.g + row % p.g) * D + ci * 8;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        cp_async_16(sQ_a + t * C::kTileBytes + c * C::kChunkBytes + sw128(row, ci),
                    valid ? src + c * 64 : p.q, valid ? 16u : 0u);
    }
  }
  cp_async_commit();
  }
  // ---- K/V codes in units u = kUnits * tile + part (rows kUnitRows * part
  // ..): 16-byte chunk rc of rows rrow + kRawRowStep * i < kUnitRows
  const int rc = ptid % C::kRawChunks, rrow = ptid / C::kRawChunks;
  const int32_t* rtt =
      kGroup ? p.req_to_token + (int64_t)p.req_pool_idx[p.members[mbeg]] * p.rtt_stride +
                   p.group_start[r]
             : p.req_to_token + (int64_t)p.req_pool_idx[r] * p.rtt_stride;
  // position of row `row` of block b in the row of req_to_token, or -1 when
  // the row holds no key (past the prefix, or past this CTA's last query)
  auto key_pos = [&](int b, int row) {
    if (b < nb_pre) {
      const int pos = b * BN + row;
      return pos < pfx ? pos : -1;
    }
    const int j = (b - nb_pre) * BN + row;
    return j < q_end ? pfx + j : -1;
  };
  // the slots of this thread's rows of the next block are loaded one block
  // ahead (registers), -1 where the row holds no key
  int32_t slot_cur[C::kUnits][C::kRawRows], slot_next[C::kUnits][C::kRawRows];
  auto load_slots = [&](int b, int32_t (&dst)[C::kUnits][C::kRawRows]) {
#pragma unroll
    for (int h = 0; h < C::kUnits; ++h) {
#pragma unroll
      for (int i = 0; i < C::kRawRows; ++i) {
        const int rr = rrow + C::kRawRowStep * i;
        const int pos = rr < C::kUnitRows ? key_pos(b, C::kUnitRows * h + rr) : -1;
        dst[h][i] = pos >= 0 ? rtt[pos] : -1;
      }
    }
  };
  if (nb > 0) load_slots(0, slot_next);
  auto issue_raw = [&](int u) {
    if (u < 2 * C::kUnits * nb) {
      const int tile = u / C::kUnits, part = u % C::kUnits;
      const int b = tile >> 1, is_v = tile & 1;
      if (!is_v && !part) {
#pragma unroll
        for (int h = 0; h < C::kUnits; ++h)
#pragma unroll
          for (int i = 0; i < C::kRawRows; ++i) slot_cur[h][i] = slot_next[h][i];
        if (b + 1 < nb) load_slots(b + 1, slot_next);
      }
      const uint8_t* pool = is_v ? p.pool_v8 : p.pool_k8;
      const uint32_t dst0 = sRaw_a + (u % C::kRaw) * C::kRawTileBytes + rc * 16;
#pragma unroll
      for (int i = 0; i < C::kRawRows; ++i) {
        const int rr = rrow + C::kRawRowStep * i;
        if (rr >= C::kUnitRows) break;
        const int32_t slot = slot_cur[part][i];
        const bool valid = slot >= 0;
        const uint8_t* src = pool + ((int64_t)(valid ? slot : 0) * p.Hkv + kvh) * D + rc * 16;
        cp_async_16(dst0 + rr * D, src, valid ? 16u : 0u);
      }
    }
    cp_async_commit();  // one group per unit (an empty one past the last)
  };
#pragma unroll
  for (int u = 0; u < C::kRaw; ++u) issue_raw(u);
  if constexpr (!q_by_softmax<true, kGroup>()) {
  // ---- widen Q in place once its group has landed (the units' groups may not)
  cp_async_wait<C::kRaw>();
#pragma unroll
  for (int t = 0; t < 2; ++t) {
#pragma unroll
    for (int i = 0; i < R::kRowsPerThread; ++i) {
      const int row = rbase + R::kRowStep * i;
      if (row >= 128) break;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const uint32_t a = sQ_a + t * C::kTileBytes + c * C::kChunkBytes + sw128(row, ci);
        const uint4 w = ld_shared_v4(a);
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
        uint32_t h[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          h[k] = pack_f16x2(__uint_as_float(x[k] << 16), __uint_as_float(x[k] & 0xFFFF0000u));
        st_shared_v4(a, h[0], h[1], h[2], h[3]);
      }
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(&bars->q_full);
  }
  // ---- widen every K/V tile into the ring, unit by unit
  bool ok = true;
  for (int tile = 0; tile < 2 * nb && ok; ++tile) {
    const int stage = tile % C::kStages, round = tile / C::kStages;
    if (round > 0) {
      ok = warp_wait(&bars->kv_empty[stage], (round - 1) & 1, bars, p);
      if (!ok) break;
    }
    // codes 16 rc .. 16 rc + 15 of a row are f16 columns of 128-byte chunk
    // rc / 4, 16-byte pieces 2 (rc % 4) and 2 (rc % 4) + 1.  Plain loads and
    // stores (not volatile asm) let the compiler issue all of a unit's loads
    // before the first store; the memory-clobbering cp.async wait above and
    // copy issue / proxy fence below keep them in place.
    uint8_t* dst0 = sKV + stage * C::kTileBytes + (rc >> 2) * C::kChunkBytes;
    const int piece = 2 * (rc & 3);
#pragma unroll
    for (int part = 0; part < C::kUnits; ++part) {
      const int u = C::kUnits * tile + part;
      cp_async_wait<C::kRaw - 1>();  // this thread's codes of unit u have landed
      const uint8_t* src0 = sRaw + (u % C::kRaw) * C::kRawTileBytes + rc * 16;
      constexpr int kBatch = kFp8Batch;  // loads in flight per thread
#pragma unroll
      for (int i0 = 0; i0 < C::kRawRows; i0 += kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int rr = rrow + C::kRawRowStep * (i0 + j);
          if (i0 + j < C::kRawRows && rr < C::kUnitRows)
            w[j] = *reinterpret_cast<const uint4*>(src0 + rr * D);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int rr = rrow + C::kRawRowStep * (i0 + j);
          if (i0 + j >= C::kRawRows || rr >= C::kUnitRows) break;
          const int row = C::kUnitRows * part + rr;
          uint4 lo, hi;
          e4m3x4_to_f16x2_scaled(w[j].x, lo.x, lo.y);
          e4m3x4_to_f16x2_scaled(w[j].y, lo.z, lo.w);
          e4m3x4_to_f16x2_scaled(w[j].z, hi.x, hi.y);
          e4m3x4_to_f16x2_scaled(w[j].w, hi.z, hi.w);
          *reinterpret_cast<uint4*>(dst0 + sw128(row, piece)) = lo;
          *reinterpret_cast<uint4*>(dst0 + sw128(row, piece + 1)) = hi;
        }
      }
      issue_raw(u + C::kRaw);
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars->kv_full[stage]);
  }
  cp_async_wait_all();  // nothing of this CTA's shared memory is still being written
}

// One CTA's work.  Extend mode: (request, KV head, two Q tiles of suffix
// tokens), keys = the request's prefix from the pool, then its suffix,
// causally; the normalised output is written as bf16.  Group mode: (shared
// group, KV head, two Q tiles of the group's member requests), whose rows are
// the members' decode queries and whose keys are the group's positions read
// once from the first member's row; each row's fp32 softmax state (reference
// max, row sum, unnormalised P.V) is written for the decode combine to merge.
//
// (bx, by, bz) name the tile: x the pair of Q tiles, y the KV head, z the
// request or group.  kPersistent: a CTA that runs tile after tile (the mixed
// batch kernel) allocates TMEM once for all of them and has initialised the
// barriers before its first tile; each tile then invalidates and initialises
// them again (the previous tile ended with every thread past its final
// barrier, every copy landed and every MMA drained).
template <int D, bool kGroup, bool kFp8, int kTiles = 2, bool kPersistent = false>
SGL_DEV void attend_tiles(const Params& p, int bx, int by, int bz) {
  using C = Cfg<D, kFp8, kTiles>;
  using R = Roles<kFp8, kTiles>;
  constexpr uint32_t kTmemCols = tmem_cols<kTiles>();
  uint8_t* smem = smem_base();
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kTiles * C::kTileBytes;
  uint8_t* sRaw = sKV + C::kStages * C::kTileBytes;
  Bars* bars = bars_of<D, kFp8, kTiles>(smem);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr bool kQSoft = q_by_softmax<kFp8, kGroup>();
  constexpr int kQThreads = kQSoft ? R::kSoftmaxWarps * 32 : R::kProducerThreads;  // q_full arrivals
  // r: the request (extend mode) or the group (group mode); the "tokens" of
  // the Q tiles are the request's suffix tokens or the group's members
  const int r = bz, kvh = by;
  const int mbeg = kGroup ? p.member_off[r] : 0;
  const int e = kGroup ? p.member_off[r + 1] - mbeg : p.extend_lens[r];
  const int q0 = bx * kTiles * p.tpt;                         // first token of this tile
  const int pfx = kGroup ? p.group_len[r] : p.prefix_lens[r];  // keys read from the pool
  const int q_end = min(e, q0 + kTiles * p.tpt);
  const int nb_pre = (pfx + BN - 1) / BN;
  const int nb = nb_pre + (kGroup ? 0 : (q_end + BN - 1) / BN);
  // Group mode: Q tile 1 holds no member (a cascade group of at most tpt
  // members, most groups of a tree): its MMAs and softmax are skipped and tile
  // 0 runs alone (tree cascade +4-5%).  Extend mode keeps both tiles: the
  // branches cost the long extend CTAs ~1%.
  const bool two_tiles = kTiles == 2 && (kGroup ? q0 + p.tpt < e : true);
  if (q0 >= e || nb <= 0) return;  // nothing to do (uniform across the CTA)

  // exclusive prefix sum of extend_lens: where request r's rows start
  if constexpr (!kGroup) {
    int32_t part = 0;
    for (int i = tid; i < r; i += (int)blockDim.x) part += p.extend_lens[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) bars->red[warp] = part;
  }
  if (tid == 0) {
    if constexpr (kPersistent) invalidate_barriers<C::kStages>(bars);
    mbar_init(&bars->q_full, kQThreads);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_ready[t], R::kSoftmaxWarps / kTiles * 32);  // the softmax warps of the tile
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->drain, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], R::kProducerThreads);
      mbar_init(&bars->kv_empty[s], 1);
    }
    bars->abort = 0;
    mbar_fence_init();
  }
  if (!kPersistent && warp == R::kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  int32_t off = 0;
  if constexpr (!kGroup) {
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) off += bars->red[w];
  }
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sQ_a = smem_u32(sQ), sKV_a = smem_u32(sKV);

  if constexpr (R::kSplitRegs && !kPersistent) {
    // every warp of a warpgroup changes its registers together (the softmax
    // warpgroups up, the others down); the kernel is built at kLaunchRegs a
    // thread (checked by the launcher)
    static_assert(R::kSoftmaxWarps % 4 == 0 && (R::kMmaWarp + 1) % 4 == 0, "whole warpgroups");
    static_assert(R::kSoftmaxWarps * R::kSoftmaxRegs + (R::kMmaWarp + 1 - R::kSoftmaxWarps) * R::kOtherRegs <=
                      (R::kMmaWarp + 1) * R::kLaunchRegs, "register split within the launch's registers");
    static_assert((R::kMmaWarp + 1) * 32 * R::kLaunchRegs <= 65536, "launch registers fit the SM");
    if (warp < R::kSoftmaxWarps)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R::kSoftmaxRegs));
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kOtherRegs));
  }
  if (R::kFullRows && warp < R::kSoftmaxWarps) {
    if constexpr (R::kFullRows) {
    // ------------------------------------------------------------ softmax (whole rows)
    if constexpr (kQSoft)
      load_q_tiles<D, kGroup, kFp8, kTiles>(p, sQ_a, &bars->q_full, tid, kQThreads, kvh, e, mbeg, q0, off);
    // warp w: Q tile t = w / 4, TMEM lane quarter q = w % 4 (rows 32q..);
    // every thread owns one row: all 128 keys of a block, all D columns of O.
    // A row whose block sum breaks the bound moves its own reference (the
    // warp reloads S and rescales O together, rows keeping their reference
    // recompute the same P with alpha = 1), so no two warps ever agree on
    // anything.
    const int t = warp >> 2, q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(t);
    const uint32_t tO = tmem + lane_off + col_o<kTiles>(t);
    const int tok = q0 + t * p.tpt + row / p.g;
    const bool row_valid = row < p.rows_used && tok < e;
    const int tok_i = row_valid ? tok : (1 << 30);  // padding rows see every key
    const float2 sc = make_float2(p.scale_log2, p.scale_log2);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = t == 0 || two_tiles;  // an empty tile's warps only meet the final barrier
    for (int b = 0; b < nb && ok; ++b) {
      if (!warp_wait(&bars->s_full[t], b & 1, bars, p)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // visible keys of this block: c < limit (key index within the block)
      int limit;
      if (b < nb_pre) limit = pfx - b * BN;
      else limit = tok_i - (b - nb_pre) * BN + 1;
      limit = max(0, min(BN, limit));
      uint32_t sr[BN];
      auto load_s = [&]() {
#pragma unroll
        for (int j = 0; j < BN / 32; ++j)
          tmem_ld32(tS + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * j]));
        tmem_wait_ld();
        if (limit < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= limit) sr[c] = __float_as_uint(-INFINITY);
        }
      };
      // P of the row's 128 keys against reference m_use, packed in place
      // over sr[0..63]; returns the row sum
      auto make_p = [&](float m_use) {
        const float2 nm = make_float2(-m_use, -m_use);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const float2 x =
              ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc, nm);
          const float2 pw = make_float2(ex2(x.x), ex2(x.y));
          if (c & 1) acc1 = fadd2(acc1, pw);
          else acc0 = fadd2(acc0, pw);
          sr[c] = kFp8 ? pack_f16x2(pw.x, pw.y) : pack_bf16x2(pw.x, pw.y);
        }
        return (acc0.x + acc0.y) + (acc1.x + acc1.y);
      };
      load_s();
      float psum = 0.f, alpha = 1.f;
      bool need = b == 0;
      if (b > 0) {
        // lazy reference: accept the block while the row sum stays within
        // the bound (every weight then fits the P operand type)
        psum = make_p(m_ref);
        need = !(psum <= R::kAcceptSum);
      }
      if (__any_sync(0xffffffffu, need)) {
        if (b > 0) load_s();  // P overwrote the registers; S is still in TMEM
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < BN; c += 2)
          mq[(c >> 1) & 3] = fmax3(mq[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
        const float m_new = need ? fmaxf(m_ref, mx) : m_ref;
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
        m_ref = m_new;
        psum = make_p(m_ref == -INFINITY ? 0.f : m_ref);
        if (b > 0) {
          // O holds blocks < b: bring it to the row's reference (alpha = 1
          // for rows that kept theirs)
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
      }
#pragma unroll
      for (int j = 0; j < BN / 64; ++j)
        tmem_st32(tS + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * j]));
      l = l * alpha + psum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[t]);
    }
    if (ok) ok = warp_wait(&bars->o_done, 0, bars, p);
    if (ok) {
      tc_fence_after();
      const uint32_t smem_a = smem_u32(smem);
      if constexpr (kGroup) {
        const int rm = row_valid ? p.members[mbeg + tok] : 0;
        const int dep = p.group_depth[r];
        const bool wr = row_valid && rm >= 0 && rm < p.batch && dep >= 0 && dep < p.max_depth;
        const int64_t ent =
            ((p.part_base + (int64_t)rm * p.max_depth + dep) * p.Hkv + kvh) * p.g + row % p.g;
        const float os = kFp8 ? p.o_scale : 1.f;
        float* dst = p.part_acc + ent * D;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * j, o);
          tmem_wait_ld();
          if (wr) {
            float4* d4 = reinterpret_cast<float4*>(dst + 32 * j);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              d4[v] = make_float4(__uint_as_float(o[4 * v]) * os, __uint_as_float(o[4 * v + 1]) * os,
                                  __uint_as_float(o[4 * v + 2]) * os, __uint_as_float(o[4 * v + 3]) * os);
          }
        }
        if (wr) p.part_ml[ent] = make_float2(m_ref, l);
      } else {
        const float inv = l > 0.f ? (kFp8 ? p.o_scale : 1.f) / l : 0.f;
        constexpr int kStride = out_stride<D>();
        const uint32_t stage = smem_a + t * 128 * kStride;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * j, o);
          tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            st_shared_v4(stage + row * kStride + 64 * j + 16 * v, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                         w[4 * v + 3]);
        }
        warp_store_rows<2 * D, kStride>(stage, q * 32, [&](int rr) -> uint8_t* {
          const int tk = q0 + t * p.tpt + rr / p.g;
          if (rr >= p.rows_used || tk >= e) return nullptr;
          return reinterpret_cast<uint8_t*>(p.out +
                                            ((int64_t)(off + tk) * p.Hq + (int64_t)kvh * p.g + rr % p.g) * D);
        });
      }
    }
    }
  } else if (warp < R::kSoftmaxWarps) {
    if constexpr (!R::kFullRows) {
    // ------------------------------------------------------------ softmax
    if constexpr (kQSoft)
      load_q_tiles<D, kGroup, kFp8, kTiles>(p, sQ_a, &bars->q_full, tid, kQThreads, kvh, e, mbeg, q0, off);
    // warp w: Q tile t, key-column half h, TMEM lane quarter q (rows 32q..)
    const int t = (warp >> 2) % kTiles, h = warp / (4 * kTiles), q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t tS = tmem + lane_off + col_s(t);
    const uint32_t tO = tmem + lane_off + col_o<kTiles>(t);
    const uint32_t pair_bar = 1 + t * 4 + q;  // named barrier of the two halves of these rows
    float* xchg_mine = &bars->xchg[t][h][row];
    const float* xchg_other = &bars->xchg[t][h ^ 1][row];
    const int tok = q0 + t * p.tpt + row / p.g;
    const bool row_valid = row < p.rows_used && tok < e;
    const int tok_i = row_valid ? tok : (1 << 30);  // padding rows see every key
    const float2 sc = make_float2(p.scale_log2, p.scale_log2);
    float m_ref = -INFINITY, l = 0.f;  // l: this half's share of the row sum
    bool ok = t == 0 || two_tiles;  // an empty tile's warps only meet the barriers
    for (int b = 0; b < nb && ok; ++b) {
      const bool ok_w = warp_wait(&bars->s_full[t], b & 1, bars, p);
      tc_fence_after();
      // visible keys of this block: c < limit (key index within the block)
      int limit;
      if (b < nb_pre) limit = pfx - b * BN;
      else limit = tok_i - (b - nb_pre) * BN + 1;
      limit = max(0, min(BN, limit)) - 64 * h;  // relative to this half's first key
      uint32_t sr[64];
      auto load_s = [&]() {
        tmem_ld32(tS + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld();
        if (limit < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c >= limit) sr[c] = __float_as_uint(-INFINITY);
        }
      };
      // P of this half's 64 keys against reference m_use, packed as bf16
      // pairs in place over sr[0..31]; returns the half's row sum
      auto make_p = [&](float m_use) {
        const float2 nm = make_float2(-m_use, -m_use);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x =
              ffma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc, nm);
          const float2 pw = make_float2(ex2(x.x), ex2(x.y));
          if (c & 1) acc1 = fadd2(acc1, pw);
          else acc0 = fadd2(acc0, pw);
          sr[c] = kFp8 ? pack_f16x2(pw.x, pw.y) : pack_bf16x2(pw.x, pw.y);
        }
        return (acc0.x + acc0.y) + (acc1.x + acc1.y);
      };
      float psum = 0.f;
      bool need = false;
      // (after a failed wait this reads stale columns of the CTA's own TMEM;
      // the vote below then ends the loop for both halves)
      load_s();
      if (b > 0) {
        // lazy reference: accept the block while this half's row sum stays
        // within the bound (every weight then fits the P operand type)
        psum = make_p(m_ref);
        need = !(psum <= R::kAcceptSum);
      }
      // The two halves of these rows vote together (one barrier): lane 0 votes
      // "a row of this warp broke the bound", lanes 1-4 vote "this warp gave
      // up waiting".  Both halves then leave together or recompute together
      // (any row over the bound, or the first block, moves the pair to the
      // block max).  The barrier also orders both halves' S reads before
      // either writes P over S's first 64 columns.
      const bool need_w = __any_sync(0xffffffffu, need);
      const uint32_t votes =
          bar_red_popc(pair_bar, 64, (lane == 0 && need_w) || (lane >= 1 && lane <= 4 && !ok_w));
      if (votes >= 4) {
        ok = false;
        break;
      }
      const bool redo = (b == 0) || (votes & 3) != 0;
      float alpha = 1.f;
      if (redo) {
        if (b > 0) load_s();  // P overwrote the registers; S is still in TMEM
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 64; c += 2)
          mq[(c >> 1) & 3] = fmax3(mq[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
        *xchg_mine = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        named_bar_sync(pair_bar, 64);
        const float mx2 = fmaxf(*xchg_mine, *xchg_other) * p.scale_log2;
        named_bar_sync(pair_bar, 64);  // both read before the buffer is reused
        const float m_new = fmaxf(m_ref, mx2);
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
        m_ref = m_new;
        psum = make_p(m_ref == -INFINITY ? 0.f : m_ref);
      }
      tmem_st32(tS + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      l = l * alpha + psum;
      if (b > 0 && redo) {
        // O (this half's D/2 columns) holds blocks < b: bring it to the new reference
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + (D / 2) * h + 32 * j, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st32(tO + (D / 2) * h + 32 * j, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_ready[t]);
    }
    if (ok) ok = warp_wait(&bars->o_done, 0, bars, p);
    // every softmax warp reaches this barrier exactly once (ok or not)
    *xchg_mine = l;
    named_bar_sync(pair_bar, 64);
    const float lrow = *xchg_mine + *xchg_other;
    const uint32_t smem_a = smem_u32(smem);
    if constexpr (kGroup) {
      if (ok) {
        tc_fence_after();
        // this half holds columns [h*D/2, (h+1)*D/2) of the row's state
        const int rm = row_valid ? p.members[mbeg + tok] : 0;
        const int dep = p.group_depth[r];
        const bool wr = row_valid && rm >= 0 && rm < p.batch && dep >= 0 && dep < p.max_depth;
        const int64_t ent =
            ((p.part_base + (int64_t)rm * p.max_depth + dep) * p.Hkv + kvh) * p.g + row % p.g;
        const float os = kFp8 ? p.o_scale : 1.f;
        float* dst = p.part_acc + ent * D + (D / 2) * h;
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
          uint32_t o[32];
          tmem_ld32(tO + (D / 2) * h + 32 * j, o);
          tmem_wait_ld();
          if (wr) {
            float4* d4 = reinterpret_cast<float4*>(dst + 32 * j);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              d4[v] = make_float4(__uint_as_float(o[4 * v]) * os, __uint_as_float(o[4 * v + 1]) * os,
                                  __uint_as_float(o[4 * v + 2]) * os, __uint_as_float(o[4 * v + 3]) * os);
          }
        }
        if (wr && h == 0) p.part_ml[ent] = make_float2(m_ref, lrow);
      }
    } else if (ok) {
      tc_fence_after();
      const float inv = lrow > 0.f ? (kFp8 ? p.o_scale : 1.f) / lrow : 0.f;
      // this half holds columns [h*D/2, (h+1)*D/2) of the output row
      constexpr int kStride = out_stride<D>();
      const uint32_t stage = smem_a + t * 128 * kStride + D * h;
#pragma unroll
      for (int j = 0; j < D / 64; ++j) {
        uint32_t o[32];
        tmem_ld32(tO + (D / 2) * h + 32 * j, o);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          st_shared_v4(stage + row * kStride + 64 * j + 16 * v, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                       w[4 * v + 3]);
      }
      warp_store_rows<D, kStride>(stage, q * 32, [&](int rr) -> uint8_t* {
        const int tk = q0 + t * p.tpt + rr / p.g;
        if (rr >= p.rows_used || tk >= e) return nullptr;
        return reinterpret_cast<uint8_t*>(
            p.out + ((int64_t)(off + tk) * p.Hq + (int64_t)kvh * p.g + rr % p.g) * D + (D / 2) * h);
      });
    }
    }
  } else if (warp < R::kMmaWarp) {
    // ------------------------------------------------------------ producers
    if constexpr (kFp8) {
      produce_fp8<D, kGroup>(p, sQ_a, sKV, sRaw, bars, tid - R::kSoftmaxWarps * 32, r, kvh, e, mbeg, q0, pfx,
                             q_end, nb_pre, nb, off);
    } else {
    constexpr int kRowStep = R::kRowStep, kRowsPerThread = R::kRowsPerThread;
    const int ptid = tid - R::kSoftmaxWarps * 32;
    const int ci = ptid & 7;
    const int rbase = ptid >> 3;  // rows rbase + kRowStep * i
    static_assert(kQSoft, "on bf16 pools the softmax warps load Q");
    // group mode: the group's keys are read from its first member's row
    const int32_t* rtt =
        kGroup ? p.req_to_token + (int64_t)p.req_pool_idx[p.members[mbeg]] * p.rtt_stride +
                     p.group_start[r]
               : p.req_to_token + (int64_t)p.req_pool_idx[r] * p.rtt_stride;
    int32_t slot_cur[kRowsPerThread], slot_next[kRowsPerThread];
    auto load_slots = [&](int b, int32_t (&dst)[kRowsPerThread]) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int j = b * BN + rbase + kRowStep * i;
        dst[i] = (b < nb_pre && j < pfx && rbase + kRowStep * i < BN) ? rtt[j] : -1;
      }
    };
    if (nb_pre > 0) load_slots(0, slot_next);
    bool ok = true;
    for (int tile = 0; tile < 2 * nb && ok; ++tile) {
      const int b = tile >> 1, is_v = tile & 1;
      const int stage = tile % C::kStages, round = tile / C::kStages;
      if (round > 0) {
        ok = warp_wait(&bars->kv_empty[stage], (round - 1) & 1, bars, p);
        if (!ok) break;
      }
      if (!is_v) {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) slot_cur[i] = slot_next[i];
        if (b + 1 < nb_pre) load_slots(b + 1, slot_next);
      }
      const uint32_t dst0 = sKV_a + stage * C::kTileBytes;
      if (b < nb_pre) {
        const __nv_bfloat16* pool = is_v ? p.pool_v : p.pool_k;
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) {
          const int row = rbase + kRowStep * i;
          if (row >= BN) break;  // rows of a block: kRowStep x kRowsPerThread may exceed it
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
          if (row >= BN) break;
          const int j = j0 + row;
          const bool valid = j < q_end;
          const __nv_bfloat16* src =
              base + ((int64_t)(off + (valid ? j : 0)) * p.Hkv + kvh) * D + ci * 8;
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            cp_async_16(dst0 + c * C::kChunkBytes + sw128(row, ci), src + c * 64, valid ? 16u : 0u);
        }
      }
      cp_async_mbar_arrive(&bars->kv_full[stage]);
    }
    cp_async_wait_all();  // nothing of this CTA's shared memory is still being written
    }
  } else if (warp == R::kMmaWarp && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = make_idesc_bf16(BM, BN, false, kFp8);
    constexpr uint32_t idO = make_idesc_bf16(BM, D, true, kFp8);
    // The issuing thread is the critical path: the tensor pipe idles while it
    // waits, so it polls with short probes first (it resumes as soon as the
    // phase completes) before the bounded wait.
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity, 200u)) return true;
      return mbar_wait_bounded(bar, parity, &bars->abort, p.status, p.wait_ns);
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
        umma_ts(tmem + col_o<kTiles>(t), tmem + col_s(t) + kk * 8, bd, idO, (acc || kk > 0) ? 1u : 0u);
      }
    };
    // copies landed by cp.async (generic proxy) are read by the tensor core
    // (async proxy): order them with a proxy fence after each wait
    bool ok = wait(&bars->q_full, 0);
    if (ok) {
      fence_proxy_async_smem();
      tc_fence_after();
    }
    for (int b = 0; b < nb && ok; ++b) {
      // V of the previous block, K of this one and P of tile 0, then one
      // proxy fence for both landed tiles
      const int kt = 2 * b, ks = kt % C::kStages;
      int vt = 0, vs = 0;
      if (b > 0) {
        vt = 2 * b - 1;
        vs = vt % C::kStages;
        if (!(ok = wait(&bars->kv_full[vs], (vt / C::kStages) & 1))) break;
      }
      if (!(ok = wait(&bars->kv_full[ks], (kt / C::kStages) & 1))) break;
      if (b > 0 && !(ok = wait(&bars->p_ready[0], (b - 1) & 1))) break;
      fence_proxy_async_smem();
      tc_fence_after();
      if (b > 0) {
        issue_pv(0, vs, b > 1);
      }
      issue_s(0, ks);
      umma_commit(&bars->s_full[0]);
      if (b > 0) {
        if (two_tiles) {
          if (!(ok = wait(&bars->p_ready[1], (b - 1) & 1))) break;
          tc_fence_after();
          issue_pv(1, vs, b > 1);
        }
        umma_commit(&bars->kv_empty[vs]);
      }
      if (two_tiles) {
        issue_s(1, ks);
        umma_commit(&bars->s_full[1]);
      }
      umma_commit(&bars->kv_empty[ks]);
    }
    if (ok) {
      const int vt = 2 * nb - 1, vs = vt % C::kStages;
      ok = wait(&bars->p_ready[0], (nb - 1) & 1) && wait(&bars->kv_full[vs], (vt / C::kStages) & 1);
      if (ok) {
        fence_proxy_async_smem();
        tc_fence_after();
        issue_pv(0, vs, nb > 1);
        if (two_tiles) ok = wait(&bars->p_ready[1], (nb - 1) & 1);
        if (ok) {
          if (two_tiles) {
            tc_fence_after();
            issue_pv(1, vs, nb > 1);
          }
          umma_commit(&bars->kv_empty[vs]);
          umma_commit(&bars->o_done);
        }
      }
    }
    // every MMA issued so far finishes before TMEM is released: after a
    // wait gave up here, and also when a softmax warp gave up waiting for
    // o_done while the last P.V MMAs were still running (the default limit:
    // the tensor core always finishes)
    umma_commit(&bars->drain);
    mbar_wait_bounded(&bars->drain, 0, nullptr, nullptr);
  }
  // no copy into this CTA's shared memory is still in flight when it exits
  // (the Q tiles' copies of warps that gave up waiting)
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if (!kPersistent && warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kFp8>
__global__ void __launch_bounds__(Roles<kFp8>::kThreads, 1) extend_kernel(Params p) {
  attend_tiles<D, false, kFp8>(p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// one Q tile: two CTAs an SM (11 warps a CTA are allocated registers as 12,
// which leaves 80 registers a thread)
template <int D, bool kFp8, int kTiles>
__global__ void __launch_bounds__(Roles<kFp8, kTiles>::kThreads, 3 - kTiles) cascade_group_kernel(Params p) {
  attend_tiles<D, true, kFp8, kTiles>(p, blockIdx.x, blockIdx.y, blockIdx.z);
  // launched dependent on the decode split kernel, whose tail items it does
  // not read: it ends only once that kernel has, so the combine launched
  // after it finds both kernels' partial states
  grid_dep_wait();
}

// The kernel parameters of an extend call (host checks of the shapes the
// kernels are built for first).
inline sgl_status make_extend_params(const ExtendArgs& a, Params* out) {
  const int g = a.num_q_heads / a.num_kv_heads;
  if (g < 1 || g > BM) return SGL_ERR_UNSUPPORTED;
  if (a.batch > 65535 || a.num_kv_heads > 65535) return SGL_ERR_UNSUPPORTED;
  Params prm = {};
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  prm.pool_k = static_cast<const __nv_bfloat16*>(a.pool_k);
  prm.pool_v = static_cast<const __nv_bfloat16*>(a.pool_v);
  prm.pool_k8 = static_cast<const uint8_t*>(a.pool_k);
  prm.pool_v8 = static_cast<const uint8_t*>(a.pool_v);
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
  // e4m3: scores in units of the widened codes (code * 2^-8) times the K
  // scale; the output takes the V scale and the 2^8 back
  prm.scale_log2 = a.sm_scale * 1.4426950408889634f * (a.kv_fp8 ? a.k_scale * kFp8Operand : 1.f);
  prm.o_scale = a.kv_fp8 ? a.v_scale * kFp8Operand : 1.f;
  prm.status = static_cast<int*>(a.workspace);
  prm.wait_ns = device_wait_limit_ns();
  *out = prm;
  return SGL_OK;
}

}  // namespace
}  // namespace ext
}  // namespace sgl
