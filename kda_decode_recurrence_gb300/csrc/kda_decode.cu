// kda_decode.cu -- the KDA decode recurrence over a slot-indexed state pool.
//
// Operation ("KdaDecode": Tensor Shapes, Default parameters; "Delta-rule
// write": the naive recurrent loop): for each request b and value head hv the
// fp32 [128, 128] state tile state_pool[state_indices[b], hv] is advanced over
// the request's tokens by decay -> delta write -> read, and written back.
//
// GB300 design (HBM-bound: 64 KiB in + 64 KiB out per tile, ~1 flop/byte):
//   * a persistent grid, two 256-thread CTAs per SM (128 registers each, so
//     16 warps per SM hide each other's latency); CTA c takes the (request,
//     value head) work items c, c + G, c + 2G, ... (G = grid size), except in
//     the multi-token instance, which deals the items ordered by request
//     length in a serpentine so that every CTA gets the same work;
//   * each tile is fetched with one 64 KiB bulk copy (cp.async.bulk, the
//     non-tensor TMA path) into the CTA's shared-memory slot as soon as the
//     previous tile has moved into registers, so the next tile is in flight
//     while the CTA computes (two per SM); an mbarrier carries the copy's
//     byte count, and every item arrives on it (with zero bytes when it has
//     no tile to fetch) so its phases advance uniformly;
//   * the tile moves from shared memory into registers once and stays there
//     across all of the request's tokens: warp w owns value columns
//     [16w, 16w + 16); lane = (row group rg 0..7, column quad cg 0..3) holds
//     rows rg, rg + 8, ..., rg + 120 of its four columns (16 float4);
//   * the k- and q-contractions over the 128 key rows are in-thread sums over
//     16 rows followed by three xor-shuffles across the 8 row groups;
//   * the first token's raw inputs (q, k, v, gate, dt_bias, beta, A_log) of
//     the next item are copied by warp 0 with cp.async into a small shared
//     buffer while the current item computes; the copies complete on an
//     mbarrier, and each warp then builds its own copy of the token's vectors
//     (normalised q and k, exp(g), beta * k, v, beta * q.k) in a private
//     shared-memory record while the tile is in flight; later tokens of an
//     item are staged 8 at a time, one warp per token, between two CTA
//     barriers.  When some request has more than one token (T > B) the
//     multi-token instance runs: warp 0's copies then bring the next item's
//     first 9 tokens (the first token and the first round of later ones)
//     into the shared buffer, so that round reads shared memory instead of
//     waiting on global loads; its refill for the item after waits until
//     that round is staged;
//   * the advanced tile is written back from registers with 128-bit
//     streaming stores;
//   * in the multi-token instance every item's descriptor (slot, token
//     range) is read from global memory once, at kernel start, into a shared
//     table (up to kMaxDesc items per CTA), so no step on an item's path waits
//     on a descriptor load (the single-token instances, bound by HBM, keep
//     their loads: the table's registers slowed them);
//   * transposed (V-first) tiles keep the same warp-to-column split, but each
//     lane holds runs of 4 consecutive rows of its columns (the tile is
//     contiguous along k there), with the token record laid out by field, so
//     their loads and stores stay 128-bit and bank-conflict-free too.
//
// The read uses q^T S_new = q^T (D S) + beta (q.k) u with u = v - k^T (D S),
// which is the same quantity as reading after the write, with one pass over
// the tile per token instead of two.
#include <type_traits>

#include "kda_async.cuh"
#include "kda_recurrence.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBufs = 1;  // tiles in flight per CTA
constexpr int kCtasPerSm = 2;
constexpr uint32_t kTileBytes = kHeadDim * kHeadDim * sizeof(float);
constexpr float kL2Eps = 1e-6f;

// One token's inputs for the 4 key rows (and 4 value columns) a lane stages.
struct TokenIn {
  uint2 q, k, v;      // 4 bf16 each
  float4 raw, bias;   // raw gate and dt_bias
  float beta_logit, a_log;
};

__device__ __forceinline__ TokenIn fetch_token(const DecodeArgs& p, int t, int h, int hv, int lane) {
  const int r0 = lane * 4;
  if (!kda_in_bounds(t >= 0 && t < p.T && h >= 0 && h < p.H && hv >= 0 && hv < p.HV, p.dev_status))
    return TokenIn{};
  TokenIn in;
  in.q = __ldg(reinterpret_cast<const uint2*>(p.q + ((size_t)t * p.H + h) * kHeadDim + r0));
  in.k = __ldg(reinterpret_cast<const uint2*>(p.k + ((size_t)t * p.H + h) * kHeadDim + r0));
  in.v = __ldg(reinterpret_cast<const uint2*>(p.v + ((size_t)t * p.HV + hv) * kHeadDim + r0));
  in.raw = __ldg(reinterpret_cast<const float4*>(p.raw_gate + ((size_t)t * p.HV + hv) * kHeadDim + r0));
  in.bias = __ldg(reinterpret_cast<const float4*>(p.dt_bias + (size_t)hv * kHeadDim + r0));
  in.beta_logit = __ldg(p.beta_logits + (size_t)t * p.HV + hv);
  in.a_log = __ldg(p.a_log + hv);
  return in;
}

// The first token of the next work item, copied asynchronously (cp.async,
// warp 0) into a small shared buffer while the current item computes: q, k,
// v rows in 8-byte pieces (the C ABI guarantees 8-byte alignment for them),
// the raw gate and dt_bias rows in 16-byte pieces, beta and A_log.
struct RawToken {
  uint2 q[32], k[32], v[32];
  float4 raw[32], bias[32];
  float beta_logit, a_log;
  float pad[2];
};

__device__ __forceinline__ void cp_async_raw(void* dst, const void* src, int bytes) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
  else if (bytes == 8)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}

// One warp, lane `lane`: the copies of token t (key head h, value head hv)
// into rt.
__device__ __forceinline__ void copy_raw_token(const DecodeArgs& p, RawToken* rt, int t, int h,
                                               int hv, int lane) {
  if (!kda_in_bounds(t >= 0 && t < p.T && h >= 0 && h < p.H && hv >= 0 && hv < p.HV, p.dev_status))
    return;
  const int r0 = lane * 4;
  cp_async_raw(&rt->q[lane], p.q + ((size_t)t * p.H + h) * kHeadDim + r0, 8);
  cp_async_raw(&rt->k[lane], p.k + ((size_t)t * p.H + h) * kHeadDim + r0, 8);
  cp_async_raw(&rt->v[lane], p.v + ((size_t)t * p.HV + hv) * kHeadDim + r0, 8);
  cp_async_raw(&rt->raw[lane], p.raw_gate + ((size_t)t * p.HV + hv) * kHeadDim + r0, 16);
  cp_async_raw(&rt->bias[lane], p.dt_bias + (size_t)hv * kHeadDim + r0, 16);
  if (lane == 0) {
    cp_async_raw(&rt->beta_logit, p.beta_logits + (size_t)t * p.HV + hv, 4);
    cp_async_raw(&rt->a_log, p.a_log + hv, 4);
  }
}

// The same without the per-head rows (dt_bias, A_log), which the
// multi-token schedule copies once per item (copy_raw_head).
__device__ __forceinline__ void copy_raw_token_rows(const DecodeArgs& p, RawToken* rt, int t,
                                                    int h, int hv, int lane) {
  if (!kda_in_bounds(t >= 0 && t < p.T && h >= 0 && h < p.H && hv >= 0 && hv < p.HV, p.dev_status))
    return;
  const int r0 = lane * 4;
  cp_async_raw(&rt->q[lane], p.q + ((size_t)t * p.H + h) * kHeadDim + r0, 8);
  cp_async_raw(&rt->k[lane], p.k + ((size_t)t * p.H + h) * kHeadDim + r0, 8);
  cp_async_raw(&rt->v[lane], p.v + ((size_t)t * p.HV + hv) * kHeadDim + r0, 8);
  cp_async_raw(&rt->raw[lane], p.raw_gate + ((size_t)t * p.HV + hv) * kHeadDim + r0, 16);
  if (lane == 0) cp_async_raw(&rt->beta_logit, p.beta_logits + (size_t)t * p.HV + hv, 4);
}
__device__ __forceinline__ void copy_raw_head(const DecodeArgs& p, RawToken* rt, int hv, int lane) {
  cp_async_raw(&rt->bias[lane], p.dt_bias + (size_t)hv * kHeadDim + lane * 4, 16);
  if (lane == 0) cp_async_raw(&rt->a_log, p.a_log + hv, 4);
}

// This thread's arrival on `bar`, once all of its earlier cp.async copies
// have completed.
__device__ __forceinline__ void arrive_after_copies(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ TokenIn read_raw_token(const RawToken* rt, int lane) {
  TokenIn in;
  in.q = rt->q[lane];
  in.k = rt->k[lane];
  in.v = rt->v[lane];
  in.raw = rt->raw[lane];
  in.bias = rt->bias[lane];
  in.beta_logit = rt->beta_logit;
  in.a_log = rt->a_log;
  return in;
}

// Build the warp's token record: L2 norms (warp reductions), the scaled
// query, the gate and decay exp(g), beta and beta * (qh . kh).  Stage is
// TokenStage (row-major tiles) or TokenStageT (transposed tiles).
template <class Stage>
__device__ __forceinline__ void build_stage(const DecodeArgs& p, const TokenIn& in, Stage& ts,
                                            int lane) {
  const int r0 = lane * 4;
  const float q[4] = {bf16_lo(in.q.x), bf16_hi(in.q.x), bf16_lo(in.q.y), bf16_hi(in.q.y)};
  const float k[4] = {bf16_lo(in.k.x), bf16_hi(in.k.x), bf16_lo(in.k.y), bf16_hi(in.k.y)};
  float qq = 0.f, kk = 0.f, qk = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    qq = fmaf(q[i], q[i], qq);
    kk = fmaf(k[i], k[i], kk);
    qk = fmaf(q[i], k[i], qk);
  }
  qq = warp_sum(qq);
  kk = warp_sum(kk);
  qk = warp_sum(qk);
  const float qs = p.q_scale * rsqrtf(qq + kL2Eps);
  const float ks = rsqrtf(kk + kL2Eps);
  const float beta = sigmoidf_(in.beta_logit);
  const float a_exp = expf(in.a_log);
  const float xr[4] = {in.raw.x + in.bias.x, in.raw.y + in.bias.y, in.raw.z + in.bias.z,
                       in.raw.w + in.bias.w};
  if constexpr (std::is_same<Stage, TokenStageT>::value) {
    float dec[4], kh[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float g = (p.gate_mode == KDA_GATE_SOFTPLUS) ? -a_exp * softplusf_(xr[i])
                                                          : p.lower_bound * sigmoidf_(a_exp * xr[i]);
      dec[i] = expf(g);
      kh[i] = k[i] * ks;
    }
    ts.decay[lane] = make_float4(dec[0], dec[1], dec[2], dec[3]);
    ts.kh[lane] = make_float4(kh[0], kh[1], kh[2], kh[3]);
    ts.qh[lane] = make_float4(q[0] * qs, q[1] * qs, q[2] * qs, q[3] * qs);
    ts.bkh[lane] = make_float4(beta * kh[0], beta * kh[1], beta * kh[2], beta * kh[3]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float g = (p.gate_mode == KDA_GATE_SOFTPLUS) ? -a_exp * softplusf_(xr[i])
                                                          : p.lower_bound * sigmoidf_(a_exp * xr[i]);
      const float kh = k[i] * ks;
      ts.row[r0 + i] = RowCoef{expf(g), kh, q[i] * qs, beta * kh};
    }
  }
  *reinterpret_cast<float4*>(&ts.v[r0]) =
      make_float4(bf16_lo(in.v.x), bf16_hi(in.v.x), bf16_lo(in.v.y), bf16_hi(in.v.y));
  if (lane == 0) ts.bqk = beta * qk * qs * ks;
}

struct Item {
  int b, hv, slot, t0, t1;
  bool range_ok;  // 0 <= t0 <= t1 <= T
  bool slot_ok;   // 0 <= slot < max_slots
  __device__ __forceinline__ bool has_tile() const { return range_ok && slot_ok && t1 > t0; }
};

__device__ __forceinline__ Item load_item(const DecodeArgs& p, long long item) {
  Item d;
  d.b = (int)(item / p.HV);
  d.hv = (int)(item - (long long)d.b * p.HV);
  d.slot = __ldg(p.state_indices + d.b);
  d.t0 = __ldg(p.cu_seqlens + d.b);
  d.t1 = __ldg(p.cu_seqlens + d.b + 1);
  d.range_ok = d.t0 >= 0 && d.t1 >= d.t0 && d.t1 <= p.T;
  d.slot_ok = d.slot >= 0 && d.slot < p.max_slots;
  return d;
}

// Descriptors kept in shared memory per CTA (slot, t0, t1 and the item
// index b * HV + hv of its items j < kMaxDesc); items beyond are read from
// global memory.
constexpr int kMaxDesc = 512;
// The multi-token schedule balances its CTAs' work when B is at most this
// (every CTA ranks the requests by length at its start).
constexpr int kMaxRankB = 1024;

__device__ __forceinline__ Item make_item(const DecodeArgs& p, int4 st) {
  Item d;
  const int it = st.w;  // B * HV < 2^31 (checked on the host)
  d.b = it / p.HV;
  d.hv = it - d.b * p.HV;
  d.slot = st.x;
  d.t0 = st.y;
  d.t1 = st.z;
  d.range_ok = d.t0 >= 0 && d.t1 >= d.t0 && d.t1 <= p.T;
  d.slot_ok = d.slot >= 0 && d.slot < p.max_slots;
  return d;
}

// Item j of this CTA: from the shared table in the multi-token instance
// (which also holds its index), else global index first + j * G, from
// global memory.
template <bool kMulti>
__device__ __forceinline__ Item get_item(const DecodeArgs& p, const int4* desc, long long first,
                                         long long G, int j) {
  return kMulti && j < kMaxDesc ? make_item(p, desc[j]) : load_item(p, first + (long long)j * G);
}
__device__ __forceinline__ long long item_index(const int4* desc, long long first, long long G,
                                                int j) {
  return j < kMaxDesc ? (long long)desc[j].w : first + (long long)j * G;
}

__device__ __forceinline__ float* tile_ptr(const DecodeArgs& p, const Item& d) {
  return p.state_pool + ((size_t)d.slot * p.HV + d.hv) * (size_t)(kHeadDim * kHeadDim);
}

// Debug builds: the item's request, value head, key head and slot lie in
// their tensors (always true in other builds).
__device__ __forceinline__ bool item_in_bounds(const DecodeArgs& p, const Item& d) {
  return kda_in_bounds(d.b >= 0 && d.b < p.B && d.hv >= 0 && d.hv < p.HV && d.hv / p.G < p.H &&
                           d.slot >= 0 && d.slot < p.max_slots,
                       p.dev_status);
}

// Arrive on the ring slot for item d (global index `item`) and start its
// tile copy when it has one.
__device__ __forceinline__ void issue_item(const DecodeArgs& p, const Item& d, long long item,
                                           float* dst, uint64_t* bar) {
#if KDA_TEST_HOOKS
  if (item == p.withhold_item) return;  // test-only: this slot's phase never completes
#else
  (void)item;
#endif
  const bool copy = d.has_tile() && item_in_bounds(p, d);
  mbar_expect_tx(bar, copy ? kTileBytes : 0u);
  if (copy) bulk_load(dst, tile_ptr(p, d), kTileBytes, bar);
}

__device__ __forceinline__ float4 step(float4 (&s)[16], const TokenStage& ts, TileLane tl,
                                       TileLaneT) {
  return tile_token_step(s, ts, tl);
}
__device__ __forceinline__ float4 step(float4 (&s)[16], const TokenStageT& ts, TileLane,
                                       TileLaneT tlt) {
  return tile_t_token_step(s, ts, tlt);
}

// Output row of token t, value head hv: 4 consecutive values from column col.
template <bool kOutBf16>
__device__ __forceinline__ void store_out(const DecodeArgs& p, int t, int hv, int col, float4 o) {
  if (!kda_in_bounds(t >= 0 && t < p.T && hv >= 0 && hv < p.HV && col >= 0 && col + 4 <= kHeadDim,
                     p.dev_status))
    return;
  const size_t off = ((size_t)t * p.HV + hv) * kHeadDim + col;
  if (kOutBf16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.output) + off), pk);
  } else {
    __stcs(reinterpret_cast<float4*>(static_cast<float*>(p.output) + off), o);
  }
}

// Fill the raw buffer with item dn's first token -- in the multi-token
// schedule with its whole first round (up to kWarps tokens).  Single-token
// schedule: warp 0 copies the one token and its 32 lanes arrive on `bar`.
// Multi-token schedule: warp w copies token w, and all kThreads threads
// arrive.  Called by the threads that arrive; a no-op for an item without a
// tile (no phase: its consumers do not wait).
template <bool kMulti>
__device__ __forceinline__ void refill_raw(const DecodeArgs& p, RawToken* rawt, uint64_t* bar,
                                           const Item& dn, int warp, int lane) {
  if (!dn.has_tile()) return;
  const int h = dn.hv / p.G;
  if (kMulti) {
    // rawt[0] carries the item's dt_bias and A_log for every token
    if (warp < dn.t1 - dn.t0) copy_raw_token_rows(p, &rawt[warp], dn.t0 + warp, h, dn.hv, lane);
    if (warp == kWarps - 1) copy_raw_head(p, &rawt[0], dn.hv, lane);
  } else {
    copy_raw_token(p, rawt, dn.t0, h, dn.hv, lane);
  }
  arrive_after_copies(bar);
}

// The single-token schedule (every request has at most one token: T <= B;
// correct for any lengths).  kVFirst: tiles are stored [V, K] (row v
// contiguous over k, the layout of a transposed state); the lanes then hold
// runs of 4 rows of one column (TileLaneT, tile_t_token_step), so tile loads
// and stores stay 128-bit and conflict-free.
template <bool kVFirst, bool kOutBf16>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) kda_decode_kernel(const DecodeArgs p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* ring = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  using Stage = typename std::conditional<kVFirst, TokenStageT, TokenStage>::type;
  Stage* wstage = reinterpret_cast<Stage*>(ring + kBufs * kHeadDim * kHeadDim);
  RawToken* rawt = reinterpret_cast<RawToken*>(wstage + kWarps);
  uint64_t* bars = reinterpret_cast<uint64_t*>(rawt + 1);
  uint64_t* rawbar = bars + kBufs;  // the first-token copies (32 arrivals: warp 0's lanes)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const TileLane tl = tile_lane();
  const TileLaneT tlt = tile_lane_t();
  Stage& ts = wstage[warp];
  const long long items = (long long)p.B * p.HV;
  const long long G = gridDim.x;
  const long long first = blockIdx.x;
  const int nmine = items > first ? (int)((items - first + G - 1) / G) : 0;

  if (blockIdx.x == 0 && threadIdx.x == 0 &&
      (p.cu_seqlens[0] != 0 || p.cu_seqlens[p.B] != p.T))
    raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kBufs; ++i) mbar_init(&bars[i], 1);
    mbar_init(rawbar, 32);
    mbar_fence_init();
    for (int j = 0; j < kBufs && j < nmine; ++j)
      issue_item(p, load_item(p, first + j * G), first + j * G, ring + j * kHeadDim * kHeadDim,
                 &bars[j]);
  }
  __syncthreads();  // the barriers are initialised
  if (warp == 0 && nmine > 0) refill_raw<false>(p, rawt, rawbar, load_item(p, first), warp, lane);
  uint32_t rawphase = 0;  // fills of the first-token buffer consumed so far

  int j = 0;
  for (; j < nmine; ++j) {
    const int buf = j % kBufs;
    const Item d = load_item(p, first + (long long)j * G);
    const bool tile = d.has_tile();
    const int h = d.hv / p.G;
    // The item's first-token inputs, copied by warp 0 during the previous item.
    __syncwarp();  // the warp is done with the previous item's record
    bool raw_ok = true;
    if (tile) {
      raw_ok = mbar_wait(rawbar, rawphase & 1u, p.wait_ns);
      ++rawphase;
      build_stage(p, read_raw_token(rawt, lane), ts, lane);
    }

    const bool arrived = mbar_wait(&bars[buf], (uint32_t)(j / kBufs) & 1u, p.wait_ns);
    float4 s[16];
    if (tile && arrived) {
      const float* src = ring + buf * kHeadDim * kHeadDim;
      if constexpr (kVFirst) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            s[4 * m + c] = *reinterpret_cast<const float4*>(src + tile_t_offset(tlt, m, c));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          s[i] = *reinterpret_cast<const float4*>(src + (tl.rg + 8 * i) * kHeadDim + tl.col);
      }
    }
    // Every thread has read the slot (and built its record from the
    // first-token buffer): the slot takes the tile of item j + kBufs, the
    // buffer the next item's first token.
    if (__syncthreads_or(!arrived || !raw_ok)) break;
    if (threadIdx.x == 0 && j + kBufs < nmine)
      issue_item(p, load_item(p, first + (long long)(j + kBufs) * G),
                 first + (long long)(j + kBufs) * G, ring + buf * kHeadDim * kHeadDim, &bars[buf]);
    // Every warp has built its record from the raw buffer: warp 0 refills it
    // with the next item's first token.
    if (warp == 0 && j + 1 < nmine)
      refill_raw<false>(p, rawt, rawbar, load_item(p, first + (long long)(j + 1) * G), warp, lane);

    if (!d.range_ok) {
      if (d.hv == 0 && threadIdx.x == 0) raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
      continue;
    }
    if (!d.slot_ok) {
      if (d.slot >= p.max_slots && d.hv == 0 && threadIdx.x == 0)
        raise_status(p.dev_status, KDA_DEV_BAD_SLOT);
      const int quads = (d.t1 - d.t0) * (kHeadDim / 4);
      for (int i = threadIdx.x; i < quads; i += kThreads)
        store_out<kOutBf16>(p, d.t0 + i / (kHeadDim / 4), d.hv, (i % (kHeadDim / 4)) * 4,
                            make_float4(0.f, 0.f, 0.f, 0.f));
      continue;
    }
    if (!tile) continue;  // no tokens: the state stays bit-identical

    // First token: this warp's own record, built while the tile was in flight.
    __syncwarp();
    {
      const float4 o = step(s, ts, tl, tlt);
      if (kVFirst ? tlt.kq == 0 : tl.rg == 0)
        store_out<kOutBf16>(p, d.t0, d.hv, kVFirst ? tlt.col : tl.col, o);
    }
    // Later tokens, 8 per round: warp w stages token c0 + w into record w, then
    // every warp steps through the round's records.  (Uniform across the CTA:
    // every thread handles the same item.)
    for (int c0 = d.t0 + 1; c0 < d.t1; c0 += kWarps) {
      const int nc = min(kWarps, d.t1 - c0);
      __syncthreads();  // all warps are done with the records of the last round
      if (warp < nc) build_stage(p, fetch_token(p, c0 + warp, h, d.hv, lane), wstage[warp], lane);
      __syncthreads();
      for (int jj = 0; jj < nc; ++jj) {
        const float4 o = step(s, wstage[jj], tl, tlt);
        if (kVFirst ? tlt.kq == 0 : tl.rg == 0)
          store_out<kOutBf16>(p, c0 + jj, d.hv, kVFirst ? tlt.col : tl.col, o);
      }
    }
    // The next item's first record goes into wstage[warp]: wait until every
    // warp has finished reading this item's rounds.
    if (d.t1 - d.t0 > 1) __syncthreads();
    if (item_in_bounds(p, d)) {
      float* dst = tile_ptr(p, d);
      if constexpr (kVFirst) {
        tile_t_store(dst, s, tlt);
      } else {
        tile_store(dst, s, tl);
      }
    }
  }

  if (j < nmine) {
    // A ring wait gave up: record it and let the copies already issued land
    // (bounded) before the CTA's shared memory is released.
    if (threadIdx.x == 0) {
      raise_status(p.dev_status, KDA_DEV_TIMEOUT);
      for (int k = j; k < j + kBufs && k < nmine; ++k)
        mbar_wait(&bars[k % kBufs], (uint32_t)(k / kBufs) & 1u, p.wait_ns);
      if (rawphase > 0) mbar_wait(rawbar, (rawphase - 1) & 1u, p.wait_ns);  // the last first-token fill
    }
    __syncthreads();
  }
}


// The multi-token schedule (some request has more than one token: T > B).
// Per item, the first round of tokens (up to kWarps) is copied ahead into
// the raw buffer (warp w copies token w, the last warp the item's dt_bias
// and A_log rows once; all kThreads threads arrive on its barrier) and built
// at the item's start, warp w building token w's record,
// while the tile is in flight; the CTA barrier that releases the tile slot
// also publishes the records and frees the raw buffer, which is refilled for
// the next item at once.  Every warp then steps through the round's records;
// tokens past the first round are staged 8 at a time from global memory.
// The item descriptors come from a shared table filled at kernel start.
template <bool kVFirst, bool kOutBf16>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) kda_decode_multi_kernel(const DecodeArgs p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  float* ring = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  using Stage = typename std::conditional<kVFirst, TokenStageT, TokenStage>::type;
  Stage* wstage = reinterpret_cast<Stage*>(ring + kBufs * kHeadDim * kHeadDim);
  RawToken* rawt = reinterpret_cast<RawToken*>(wstage + kWarps);  // [kWarps]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rawt + kWarps);
  uint64_t* rawbar = bars + kBufs;                    // kThreads arrivals per fill
  int4* desc = reinterpret_cast<int4*>(rawbar + 1);  // [kMaxDesc] slot, t0, t1, item

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const TileLane tl = tile_lane();
  const TileLaneT tlt = tile_lane_t();
  const long long items = (long long)p.B * p.HV;
  const long long G = gridDim.x;
  const long long first = blockIdx.x;
  // Work balance: an item costs a fixed part plus a part per token, and the
  // kernel lasts as long as its busiest CTA.  When the requests can be ranked
  // at the start (B <= kMaxRankB) and every CTA's list fits the table, the
  // items are taken in order of their request's length, longest first (ties
  // by request), and dealt to the CTAs in a serpentine: round r gives
  // position r G + i to CTA i when r is even and to CTA G - 1 - i when it is
  // odd.  Otherwise CTA c takes items c, c + G, c + 2G, ...  Which CTA
  // computes an item does not change its result.
  const bool balanced = p.B <= kMaxRankB && (items + G - 1) / G <= kMaxDesc;
  int nmine;
  if (balanced) {
    const long long R = items / G, rem = items - R * G;
    nmine = (int)R + (int)((R & 1) == 0 ? first < rem : G - 1 - first < rem);
  } else {
    nmine = items > first ? (int)((items - first + G - 1) / G) : 0;
  }

  if (blockIdx.x == 0 && threadIdx.x == 0 &&
      (p.cu_seqlens[0] != 0 || p.cu_seqlens[p.B] != p.T))
    raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
  // The requests' ranks, in the tile slot (free until the first tile is issued).
  int* len_s = reinterpret_cast<int*>(ring);  // [B] token counts
  int* order = len_s + kMaxRankB;             // [B] rank -> request
  if (balanced) {
    for (int b = threadIdx.x; b < p.B; b += kThreads)
      len_s[b] = __ldg(p.cu_seqlens + b + 1) - __ldg(p.cu_seqlens + b);
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
      const int nb = len_s[b];
      int r = 0;
      for (int b2 = 0; b2 < p.B; ++b2) {
        const int n2 = len_s[b2];
        r += (n2 > nb || (n2 == nb && b2 < b)) ? 1 : 0;
      }
      order[r] = b;
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < nmine && i < kMaxDesc; i += kThreads) {
    long long item = first + (long long)i * G;
    if (balanced) {
      const long long pos = (long long)i * G + ((i & 1) == 0 ? first : G - 1 - first);
      item = (long long)order[pos / p.HV] * p.HV + pos % p.HV;
    }
    const int b = (int)(item / p.HV);
    desc[i] = make_int4(__ldg(p.state_indices + b), __ldg(p.cu_seqlens + b),
                        __ldg(p.cu_seqlens + b + 1), (int)item);
  }
  __syncthreads();  // the descriptors are in place and the slot is free again
  if (threadIdx.x == 0) {
    for (int i = 0; i < kBufs; ++i) mbar_init(&bars[i], 1);
    mbar_init(rawbar, kThreads);
    mbar_fence_init();
    for (int j = 0; j < kBufs && j < nmine; ++j)
      issue_item(p, get_item<true>(p, desc, first, G, j), item_index(desc, first, G, j),
                 ring + j * kHeadDim * kHeadDim, &bars[j]);
  }
  __syncthreads();  // the barriers are initialised
  if (nmine > 0) refill_raw<true>(p, rawt, rawbar, get_item<true>(p, desc, first, G, 0), warp, lane);
  uint32_t rawphase = 0;  // fills of the raw buffer consumed so far

  int j = 0;
  for (; j < nmine; ++j) {
    const int buf = j % kBufs;
    const Item d = get_item<true>(p, desc, first, G, j);
    const bool tile = d.has_tile();
    const int h = d.hv / p.G;
    const int n1 = min(kWarps, d.t1 - d.t0);  // tokens of the first round
    // The first round's records, built from the raw buffer while the tile is
    // in flight (every warp finished reading the previous item's records
    // before that item's closing barrier).
    bool raw_ok = true;
    if (tile) {
      raw_ok = mbar_wait(rawbar, rawphase & 1u, p.wait_ns);
      ++rawphase;
      if (warp < n1) {
        TokenIn in = read_raw_token(&rawt[warp], lane);
        in.bias = rawt[0].bias[lane];
        in.a_log = rawt[0].a_log;
        build_stage(p, in, wstage[warp], lane);
      }
    }

    const bool arrived = mbar_wait(&bars[buf], (uint32_t)(j / kBufs) & 1u, p.wait_ns);
    float4 s[16];
    if (tile && arrived) {
      const float* src = ring + buf * kHeadDim * kHeadDim;
      if constexpr (kVFirst) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            s[4 * m + c] = *reinterpret_cast<const float4*>(src + tile_t_offset(tlt, m, c));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          s[i] = *reinterpret_cast<const float4*>(src + (tl.rg + 8 * i) * kHeadDim + tl.col);
      }
    }
    // Every thread has read the slot and every record of the round is built:
    // the slot takes the tile of item j + kBufs, the raw buffer the next
    // item's first round.
    if (__syncthreads_or(!arrived || !raw_ok)) break;
    if (threadIdx.x == 0 && j + kBufs < nmine)
      issue_item(p, get_item<true>(p, desc, first, G, j + kBufs),
                 item_index(desc, first, G, j + kBufs), ring + buf * kHeadDim * kHeadDim,
                 &bars[buf]);
    if (j + 1 < nmine)
      refill_raw<true>(p, rawt, rawbar, get_item<true>(p, desc, first, G, j + 1), warp, lane);

    if (!d.range_ok) {
      if (d.hv == 0 && threadIdx.x == 0) raise_status(p.dev_status, KDA_DEV_BAD_SEQLEN);
      continue;
    }
    if (!d.slot_ok) {
      if (d.slot >= p.max_slots && d.hv == 0 && threadIdx.x == 0)
        raise_status(p.dev_status, KDA_DEV_BAD_SLOT);
      const int quads = (d.t1 - d.t0) * (kHeadDim / 4);
      for (int i = threadIdx.x; i < quads; i += kThreads)
        store_out<kOutBf16>(p, d.t0 + i / (kHeadDim / 4), d.hv, (i % (kHeadDim / 4)) * 4,
                            make_float4(0.f, 0.f, 0.f, 0.f));
      continue;
    }
    if (!tile) continue;  // no tokens: the state stays bit-identical

    for (int jj = 0; jj < n1; ++jj) {
      const float4 o = step(s, wstage[jj], tl, tlt);
      if (kVFirst ? tlt.kq == 0 : tl.rg == 0)
        store_out<kOutBf16>(p, d.t0 + jj, d.hv, kVFirst ? tlt.col : tl.col, o);
    }
    // Tokens past the first round, 8 per round from global memory.
    for (int c0 = d.t0 + kWarps; c0 < d.t1; c0 += kWarps) {
      const int nc = min(kWarps, d.t1 - c0);
      __syncthreads();  // all warps are done with the records of the last round
      if (warp < nc) build_stage(p, fetch_token(p, c0 + warp, h, d.hv, lane), wstage[warp], lane);
      __syncthreads();
      for (int jj = 0; jj < nc; ++jj) {
        const float4 o = step(s, wstage[jj], tl, tlt);
        if (kVFirst ? tlt.kq == 0 : tl.rg == 0)
          store_out<kOutBf16>(p, c0 + jj, d.hv, kVFirst ? tlt.col : tl.col, o);
      }
    }
    if (item_in_bounds(p, d)) {
      float* dst = tile_ptr(p, d);
      if constexpr (kVFirst) {
        tile_t_store(dst, s, tlt);
      } else {
        tile_store(dst, s, tl);
      }
    }
    // The next item's records overwrite this item's: every warp must be done
    // reading them.
    __syncthreads();
  }

  if (j < nmine) {
    // A wait gave up: record it and let the copies already issued land
    // (bounded) before the CTA's shared memory is released.
    if (threadIdx.x == 0) {
      raise_status(p.dev_status, KDA_DEV_TIMEOUT);
      for (int k = j; k < j + kBufs && k < nmine; ++k)
        mbar_wait(&bars[k % kBufs], (uint32_t)(k / kBufs) & 1u, p.wait_ns);
    }
    // The last raw-buffer fill (every thread's copies arrive on it).
    if (rawphase > 0) mbar_wait(rawbar, (rawphase - 1) & 1u, p.wait_ns);
    __syncthreads();
  }
}

}  // namespace

size_t decode_smem_bytes(bool multi) {
  return 128 + (size_t)kBufs * kTileBytes + kWarps * sizeof(TokenStage) +
         (multi ? kWarps : 1) * sizeof(RawToken) + (kBufs + 1) * sizeof(uint64_t) +
         (multi ? kMaxDesc * sizeof(int4) : 0);
}

#if KDA_TEST_HOOKS
// Test-only build: the wait limit and the withheld item of the next launches.
unsigned long long g_test_wait_ns = kWaitLimitNs;
long long g_test_withhold_item = -1;
#endif

cudaError_t launch_kda_decode(const DecodeArgs& in, cudaStream_t stream) {
  DecodeArgs args = in;
  args.wait_ns = kWaitLimitNs;
  args.withhold_item = -1;
#if KDA_TEST_HOOKS
  args.wait_ns = g_test_wait_ns;
  args.withhold_item = g_test_withhold_item;
#endif
  const long long items = (long long)args.B * args.HV;
  if (items == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // The multi-token schedule when some request has more than one token.
  const bool multi = args.T > args.B;
  const size_t smem = decode_smem_bytes(multi);
  void (*kernel)(DecodeArgs) =
      multi ? (args.v_first
                   ? (args.out_bf16 ? kda_decode_multi_kernel<true, true> : kda_decode_multi_kernel<true, false>)
                   : (args.out_bf16 ? kda_decode_multi_kernel<false, true> : kda_decode_multi_kernel<false, false>))
            : (args.v_first
                   ? (args.out_bf16 ? kda_decode_kernel<true, true> : kda_decode_kernel<true, false>)
                   : (args.out_bf16 ? kda_decode_kernel<false, true> : kda_decode_kernel<false, false>));
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long slots = (long long)sms * kCtasPerSm;
  const long long grid = items < slots ? items : slots;
  kernel<<<(unsigned)grid, kThreads, smem, stream>>>(args);
  return cudaGetLastError();
}

}  // namespace kda

#if KDA_TEST_HOOKS
// Exported by the test-only build (libkda_testhooks.so), not declared in
// kda.h: set the decode kernel's wait limit and the work item (request *
// HV + value head) whose tile copy is withheld, for the launches that follow.
extern "C" void kda_test_set_decode_hooks(long long withhold_item, unsigned long long wait_ns) {
  kda::g_test_withhold_item = withhold_item;
  kda::g_test_wait_ns = wait_ns;
}
#endif
