// walk_batched.cu -- the persistent walk for large batches (and vocabularies
// too big to hold on chip): per step every CTA computes D = W2_shard @ U with
// U = [u_0 .. u_{B-1}] (256 x B) as a real dense contraction on the 5th-gen
// tensor cores -- tcgen05.mma, A = a 128-row W2 tile from shared memory,
// B = U from shared memory, N = B rounded up to 16, D in tensor memory.
// Source: "Keeping the Draft Walk on Chip: One Launch for DSpark's Markov
// Head", sections "B200: the bf16 table fits on chip" (request n is column n
// of the MMA's N operand; batching is almost free for the tensor cores) and
// "V = 248,320: 62% on chip, the rest streamed" (one thread streams W2 rows
// with TMA into a shared-memory ring and issues tcgen05 MMAs straight from
// shared memory; the ring keeps refilling across steps because W2 does not
// depend on the token).
//
// CTA = 16 epilogue warps + 1 control warp.  The control warp's lane 0 keeps
// NST half-tiles (32 KB: 128 rows x 128 K) of the CTA's W2 shard in flight
// with cp.async.bulk, issues the 8 MMAs of each half-tile into one of two
// TMEM accumulators (128 x N fp32 each), and commits them to mbarriers.  The
// epilogue warps read a finished accumulator (warp w: lane quarter w % 4,
// column quarter w / 4) 8 columns at a time, one row per lane; the bf16
// biases go through a small per-warp shared-memory buffer that turns the
// 32 x 8 block around, so that each lane then owns 8 consecutive tokens of ONE
// request: its base logits are one 16-byte load, two logits are summed per
// bf16x2 add, and one Philox call serves four of its tokens (the counter is
// shared by tokens 4j .. 4j + 3).  Keys are folded per request and the
// accumulator is freed.  After the last tile the CTA's best key per request
// goes through the atomic rendezvous and the next u rows are gathered into U.
//
// Requests are laid out in MMA columns greedy-first (a stable partition by
// temperature), so an 8-column chunk is, but for one, all greedy or all
// sampled and the lanes of a warp rarely diverge on the noise.  W2 copies
// carry an L2 evict-last policy and the base loads evict-first: W2 (re-read
// every step) then stays in L2 beside the base stream (read once).
#include "tc_ptx.cuh"
#include "walk_common.cuh"
#include "walk_kernels.h"

namespace dspark {

namespace {

constexpr int kEpiWarps = 16;                 // 4 per TMEM lane quarter
constexpr int kBatThreads = (kEpiWarps + 1) * 32;
constexpr int kStageBytes = 32768;            // half a tile: 128 rows x 128 K bf16
constexpr int kBlockBytes = 4096;             // 128 rows x 16 K
constexpr int kMaxStages = 6;
constexpr int kCW = 8;                        // accumulator columns per epilogue chunk
constexpr int kStgStride = 40;                // uint16 per column of the turn-around buffer
constexpr int kStgWarpElems = kCW * kStgStride;
constexpr int kWbCols = 64;                   // wbest slots per warp (N / 4 <= 64)

struct BatchedArgs {
  WalkArgs w;
  const uint8_t* W2b;        // per CTA: T tiles x 16 K-blocks x 4 KB (core-matrix layout)
  int R;                     // rows per CTA (multiple of 128)
  int T;                     // tiles per CTA
  int N;                     // MMA N: B rounded up to 16 (<= 256)
  int nst;                   // ring stages
  int max_B;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint64_t t0,
                                         int64_t limit) {
  uint32_t spins = 0;
  while (!ptx::mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0u && (int64_t)(globaltimer_ns() - t0) > limit) return false;
  }
  return true;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_u32(bar)) : "memory");
}

// Column c of U = W1[tok of request col2req[c]] (core matrix (kc, c / 8) at
// (kc * N/8 + c/8) * 128); columns without a request keep their zeros.
// Eight rows' chunks in flight per thread before any store.
__device__ __forceinline__ void gather_u(const WalkArgs& a, const int32_t* tok_s,
                                         const int16_t* col2req, uint8_t* U, int N) {
  const int epi_threads = kEpiWarps * 32;
  const int total = N * 32;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * epi_threads) {
    uint4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * epi_threads;
      const int r = i < total ? (int)col2req[i >> 5] : -1;
      if (r >= 0)
        x[u] = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok_s[r] * kRank) + (i & 31));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * epi_threads;
      if (i < total && col2req[i >> 5] >= 0) {
        const int b = i >> 5, c = i & 31;
        *reinterpret_cast<uint4*>(U + ((size_t)c * (N >> 3) + (b >> 3)) * 128 + (b & 7) * 16) =
            x[u];
      }
    }
  }
  ptx::fence_proxy_async_smem();
}

// Width of the column slots: 8 (one epilogue chunk) when a column quarter
// holds a multiple of 8 columns, else 4.
__device__ __forceinline__ int slot_width(int N) { return ((N >> 2) & 7) == 0 ? 8 : 4; }

// MMA column of the request with rank r (ranks: greedy requests first, each
// kind in request order).  Ranks fill slots of slot_width columns taken
// round-robin over the four column quarters (slot s: quarter s % 4, position
// s / 4 in it), so every quarter -- and thus every epilogue warp -- gets an
// even share of the sampled requests, while epilogue chunks stay of one kind
// but for at most one.  Each quarter's live columns are a prefix of it.
__device__ __forceinline__ int rank_column(int r, int N) {
  const int W = slot_width(N);
  const int s = r / W;
  return (s & 3) * (N >> 2) + (s >> 2) * W + (r - s * W);
}

// Live columns of column quarter g (a prefix of its N / 4 columns).
__device__ __forceinline__ int quarter_live(int g, int B, int N) {
  const int W = slot_width(N);
  int n = 0;
  for (int p = 0; p < (N >> 2) / W; ++p) {
    const int m = B - (p * 4 + g) * W;
    n += m <= 0 ? 0 : (m > W ? W : m);
  }
  return n;
}

// col2req[c] = request of MMA column c (-1: none).  One warp.
__device__ __forceinline__ void order_columns(int B, int N, const float* temp_s,
                                              int16_t* col2req, int lane) {
  for (int c = lane; c < 256; c += 32) col2req[c] = -1;
  __syncwarp();
  int ng = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    ng += __popc(__ballot_sync(0xFFFFFFFFu, b < B && !(temp_s[b] > 0.0f)));
  }
  int pg = 0, ps = ng;
  const unsigned below = (1u << lane) - 1u;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const bool in = b < B;
    const bool greedy = in && !(temp_s[b] > 0.0f);
    const unsigned mg = __ballot_sync(0xFFFFFFFFu, greedy);
    const unsigned ms = __ballot_sync(0xFFFFFFFFu, in && !greedy);
    if (greedy) col2req[rank_column(pg + __popc(mg & below), N)] = (int16_t)b;
    else if (in) col2req[rank_column(ps + __popc(ms & below), N)] = (int16_t)b;
    pg += __popc(mg);
    ps += __popc(ms);
  }
  __syncwarp();
}

// Base logits of tokens v0 .. v0 + 7 from one request's row of this step
// (row null: none), packed two per word; tokens at or past V read as 0.
// `vec`: one 16-byte load that skips L1 and carries the L2 `policy` (V a
// multiple of 8, 16-byte aligned base).
__device__ __forceinline__ void load_base8(const WalkArgs& a, const uint16_t* row, int64_t v0,
                                           bool vec, uint64_t policy, uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = 0u;
  if (row == nullptr) return;
  const uint16_t* src = row + v0;
  if (vec && v0 + 8 <= a.V) {
    const uint4 x = ptx::ldg_nc_na_hint(src, policy);
    w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (v0 + i < a.V) w[i >> 1] |= (uint32_t)__ldg(src + i) << (16 * (i & 1));
  }
}

// Two bf16 logits at once: bf16(base + bias), each rounded once to nearest even.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t x, uint32_t y) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
  return d;
}

// Temperatures below this take their reciprocal scaled (see gumbel8).
constexpr float kTinyT = 0x1p-120f;

// Gumbel-max scores of the 8 logits lg of tokens v0 .. v0 + 7 (request b,
// step k): fp32(logit / T) + noise where T > 0, the logit itself where T = 0.
// The quotient is the product with the rounded reciprocal, taken as
// fl(fl(logit * inv_T) * qscale + g) in one fused step: qscale = 1 and
// inv_T = fl(1/T) for T >= 2^-120; below, inv_T = fl(1/(2^64 T)) and qscale =
// 2^64.  The scalings by 2^64 are exact, so this is the product with fl(1/T)
// with the exponent range extended: the same bits wherever fl(1/T) is finite,
// and a finite reciprocal where it overflows.
__device__ __forceinline__ void gumbel8(const float (&lg)[8], float T, float inv_T, float qscale,
                                        int64_t v0, int k, int b, const PhiloxKeys& pk,
                                        float (&sc)[8]) {
  const bool sampled = T > 0.0f;
#pragma unroll
  for (int c4 = 0; c4 < 2; ++c4) {
    const uint4 r = philox4x32_10(
        make_uint4((uint32_t)(v0 >> 2) + (uint32_t)c4, (uint32_t)k, (uint32_t)b, 0u), pk);
    const uint32_t x[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float l = lg[4 * c4 + e];
      const float q = __fmul_rn(l, inv_T);
      sc[4 * c4 + e] = sampled ? __fmaf_rn(q, qscale, gumbel_noise(x[e])) : l;
    }
  }
}

// The selection key of 8 scores of tokens v0 .. v0 + 7, nvalid of them real:
// {ord32(best score), inverted id}, ties to the smallest id.
__device__ __forceinline__ unsigned long long best_key8(const float (&sc)[8], int64_t v0,
                                                        int64_t nvalid) {
  float best = sc[0];
  int best_i = 0;
  if (nvalid >= 8) {
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (sc[i] > best) { best = sc[i]; best_i = i; }
  } else {
#pragma unroll
    for (int i = 1; i < 8; ++i)
      if (i < nvalid && sc[i] > best) { best = sc[i]; best_i = i; }
  }
  return ((unsigned long long)ord32(best) << 32) |
         (unsigned long long)(0xFFFFFFFFu - (uint32_t)(v0 + best_i));
}

// bf16 logit i of the 8 packed two per word in lw, as fp32.
__device__ __forceinline__ void unpack8(const uint32_t (&lw)[4], float (&lg)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    lg[i] = __uint_as_float((i & 1) ? (lw[i >> 1] & 0xFFFF0000u) : (lw[i >> 1] << 16));
}

// Tokens v0 .. v0 + 7 of request b at step k: logit = bf16(base + bias) (the
// bias already rounded to bf16), the optional copy to out_logits, the
// selection score and the best key {order bits, inverted id}; ties keep the
// smallest id.  Tokens at or past V do not take part.  `kind` is the same for
// the whole warp: 0 = every live lane greedy (score = logit); 1 = noise drawn
// for every lane (one Philox call per four tokens) and used where T > 0;
// 2 = the group sampler (the 8 tokens are one group: group_key) where T > 0,
// greedy elsewhere.
__device__ __forceinline__ unsigned long long score8(const WalkArgs& a, const PhiloxKeys& pk,
                                                     int k, int b, float T, float inv_T,
                                                     int64_t v0, const uint4& bz,
                                                     const uint32_t (&bw)[4], bool vec,
                                                     int kind) {
  const int64_t nvalid = a.V - v0;
  if (nvalid <= 0) return 0ull;
  uint32_t lw[4];
  lw[0] = add_bf16x2(bw[0], bz.x);
  lw[1] = add_bf16x2(bw[1], bz.y);
  lw[2] = add_bf16x2(bw[2], bz.z);
  lw[3] = add_bf16x2(bw[3], bz.w);
  float lg[8];
  unpack8(lw, lg);
  if (a.out_logits != nullptr) {
    uint16_t* dst = a.out_logits + ((size_t)b * a.gamma + k) * (size_t)a.V + v0;
    if (vec && nvalid >= 8) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < nvalid) dst[i] = (uint16_t)(lw[i >> 1] >> (16 * (i & 1)));
    }
  }
  if (kind == 2 && T > 0.0f)
    return group_key(lg, nvalid < 8 ? (int)nvalid : 8, T, inv_T, (uint32_t)v0, k, b, pk);
  float sc[8];
  if (kind == 0 || kind == 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i] = lg[i];
  } else {
    gumbel8(lg, T, inv_T, T < kTinyT ? 0x1p64f : 1.0f, v0, k, b, pk, sc);
  }
  return best_key8(sc, v0, nvalid);
}

__global__ void __launch_bounds__(kBatThreads, 1) walk_batched_kernel(const BatchedArgs ba) {
  const WalkArgs& a = ba.w;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int N = ba.N;
  uint8_t* ring = smem;                                            // nst x 32 KB
  uint8_t* U = smem + (size_t)ba.nst * kStageBytes;                // N x 512 B
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(U + (size_t)N * 512);
  // wbest: [16 warps][64] running best per (warp, column in the warp's quarter)
  unsigned long long* cta_key = wbest + kEpiWarps * kWbCols;       // [256] per request
  int32_t* tok_s = reinterpret_cast<int32_t*>(cta_key + 256);      // [256] per request
  float* temp_s = reinterpret_cast<float*>(tok_s + 256);           // [256] per request
  int16_t* col2req = reinterpret_cast<int16_t*>(temp_s + 256);     // [256] per column
  float* tcol = reinterpret_cast<float*>(col2req + 256);           // [256] T per column
  float* icol = tcol + 256;                                        // [256] fl(1/T) per column
  uint16_t* stage = reinterpret_cast<uint16_t*>(icol + 256);       // [16 warps][8][40]
  // [256] per column: this step's base row of the column's request (null: none)
  const uint16_t** colbase =
      reinterpret_cast<const uint16_t**>(stage + (size_t)kEpiWarps * kStgWarpElems);
  __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t dfull[2], dempty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ int flag_s, abort_s;
  __shared__ uint32_t round_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int64_t row0 = (int64_t)cta * ba.R;
  const int T = ba.T, nst = ba.nst;
  const uint8_t* gw = ba.W2b + (size_t)cta * T * 16 * kBlockBytes;
  const bool vec = (a.V % 8 == 0) && ((reinterpret_cast<uintptr_t>(a.base) & 15u) == 0) &&
                   ((reinterpret_cast<uintptr_t>(a.out_logits) & 15u) == 0);

  const int bad = check_inputs(a, &flag_s);
  if (bad != 0) {
    if (cta == 0) {
      if (threadIdx.x == 0) set_status(a.sync.hdr, bad);
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    }
    return;
  }

  // ---------------------------------------------------------------- entry --
  trace_stamp(a, a.gamma, 0);
  if (threadIdx.x == 0) {
    round_s = *reinterpret_cast<volatile uint32_t*>(&a.sync.hdr->round);
    abort_s = 0;
    for (int i = 0; i < nst; ++i) {
      ptx::mbar_init(&full_bar[i], 1);
      ptx::mbar_init(&empty_bar[i], 1);
    }
    ptx::mbar_init(&dfull[0], 1);
    ptx::mbar_init(&dfull[1], 1);
    ptx::mbar_init(&dempty[0], kEpiWarps);
    ptx::mbar_init(&dempty[1], kEpiWarps);
    ptx::fence_mbar_init();
  }
  if (warp == kEpiWarps) {
    ptx::tmem_alloc(&tmem_base_s, 512);
    ptx::tmem_relinquish();
  }
  for (int b = threadIdx.x; b < 256; b += blockDim.x) {
    tok_s[b] = b < a.B ? a.anchor[b] : 0;
    temp_s[b] = b < a.B ? a.temperature[b] : 0.0f;
  }
  for (int i = threadIdx.x; i < N * 512 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(U)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (cta == 0) clear_other_parity(a.sync, round_s & 1u);
  if (warp == 0) order_columns(a.B, N, temp_s, col2req, lane);
  __syncthreads();
  for (int c = threadIdx.x; c < 256; c += blockDim.x) {
    const float Tc = col2req[c] >= 0 ? temp_s[col2req[c]] : 0.0f;
    tcol[c] = Tc;
    // the group sampler takes fl(1/T) (0 where it overflows); the Gumbel
    // scores take the reciprocal of 2^64 T below 2^-120 (see gumbel8)
    icol[c] = !(Tc > 0.0f)                    ? 0.0f
              : a.sampler == 1 || Tc >= kTinyT ? inv_temperature(Tc)
                                               : __frcp_rn(__fmul_rn(Tc, 0x1p64f));
    colbase[c] = col2req[c] >= 0 ? a.base + (size_t)col2req[c] * a.gamma * (size_t)a.V : nullptr;
  }
  if (warp < kEpiWarps) gather_u(a, tok_s, col2req, U, N);

  // control state (lane 0 of the control warp)
  const int stages_total = 2 * T * a.gamma;   // half-tiles consumed this round
  int issued = 0;                             // half-tiles whose copy was issued
  // W2 is re-read every step and the base logits once: W2 keeps its L2 lines
  // ahead of the base stream, which would otherwise push it out at large B
  const uint64_t w2_policy = ptx::policy_evict_last();
  if (warp == kEpiWarps && lane == 0) {
    const int pre = nst < stages_total ? nst : stages_total;
    for (; issued < pre; ++issued) {
      const int gl = issued % (2 * T);
      ptx::mbar_expect_tx(&full_bar[issued % nst], kStageBytes);
      ptx::bulk_g2s_hint(ring + (size_t)(issued % nst) * kStageBytes,
                         gw + (size_t)gl * kStageBytes, kStageBytes, &full_bar[issued % nst],
                         w2_policy);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();

  const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
                         ((uint32_t)(128 >> 4) << 24);
  const uint32_t u_addr = ptx::smem_u32(U);
  const uint32_t ring_addr = ptx::smem_u32(ring);
  bool ok = true;
  int consumed = 0;   // control: half-tiles whose MMAs were issued
  int G = 0;          // tiles processed so far this round (both roles track it)

  trace_stamp(a, a.gamma, 2);
  for (int k = 0; k < a.gamma && ok; ++k) {
    ptx::tc_fence_after();
    const uint64_t t_step = globaltimer_ns();
    trace_stamp(a, k, 0);
    if (warp == kEpiWarps) {
      // ------------------------------------------------------ control warp
      if (lane == 0) {
        for (int t = 0; t < T && ok; ++t, ++G) {
          const int d = G & 1;
          if (G >= 2 && !wait_bar(&dempty[d], (uint32_t)(((G - 2) >> 1) & 1), t_step,
                                  a.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          for (int h = 0; h < 2; ++h, ++consumed) {
            const int s = consumed % nst;
            if (!wait_bar(&full_bar[s], (uint32_t)((consumed / nst) & 1), t_step, a.timeout_ns)) {
              ok = false;
              break;
            }
            // one descriptor pair per half-tile: the start-address field (bits
            // 0..13, in 16-byte units) then advances by one 4 KB K block of A and
            // one 16-deep slice of U per MMA; shared addresses stay below 256 KB,
            // so the field never carries into the next one
            const uint64_t adesc0 =
                ptx::smem_desc_noswizzle(ring_addr + (uint32_t)s * kStageBytes, 2048, 128);
            const uint64_t bdesc0 = ptx::smem_desc_noswizzle(
                u_addr + (uint32_t)(8 * h) * 32u * (uint32_t)N, 16u * (uint32_t)N, 128);
            const uint32_t dcol = tmem + (uint32_t)(d * 256);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint64_t adesc = adesc0 + (uint64_t)(j * (kBlockBytes >> 4));
              const uint64_t bdesc = bdesc0 + (uint64_t)(j * 2 * N);
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dcol),
                  "l"(adesc), "l"(bdesc), "r"(idesc), "r"((h | j) != 0 ? 1u : 0u)
                  : "memory");
            }
            ptx::tc_commit(&empty_bar[s]);
            // refill the slot consumed one half-tile ago (its MMAs are done or nearly)
            if (consumed >= 1 && issued < stages_total) {
              const int prev = consumed - 1;
              const int ps = prev % nst;
              if (!wait_bar(&empty_bar[ps], (uint32_t)((prev / nst) & 1), t_step, a.timeout_ns)) {
                ok = false;
                break;
              }
              const int gl = issued % (2 * T);
              ptx::mbar_expect_tx(&full_bar[ps], kStageBytes);
              ptx::bulk_g2s_hint(ring + (size_t)ps * kStageBytes, gw + (size_t)gl * kStageBytes,
                                 kStageBytes, &full_bar[ps], w2_policy);
              ++issued;
            }
          }
          if (!ok) break;
          ptx::tc_commit(&dfull[d]);
        }
        if (!ok) {
          abort_round(a.sync.hdr, round_s, kStatusTimeout);
          abort_s = 1;
        }
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------- epilogue warps
      // warp w: rows 32 (w % 4) .. +31 of every tile (its TMEM lane quarter),
      // columns [c0, c0 + N / 4) with c0 = (w / 4) N / 4, 8 at a time.  After
      // the turn-around, lane (jl, hl) owns column c0 + cb + jl and rows
      // 8 hl .. 8 hl + 7 of the warp's 32; its base logits for the next chunk
      // are loaded before the current chunk is computed.
      const int q = warp & 3, grp = warp >> 2;
      const int cols = N >> 2;
      const int c0 = grp * cols;
      const int act = quarter_live(grp, a.B, N);     // this warp's live columns
      const int cpt = (act + kCW - 1) / kCW;         // chunks per tile
      const int nc = cpt * T;
      const int jl = lane & 7, hl = lane >> 3;
      uint16_t* stg = stage + warp * kStgWarpElems;
      for (int i = lane; i < kWbCols; i += 32) wbest[warp * kWbCols + i] = 0ull;
      __syncwarp();
      const uint2 eseed = round_seed(a, round_s);     // this round's Philox key
      const PhiloxKeys pk = philox_keys(eseed.x, eseed.y);
      const uint64_t base_policy = ptx::policy_evict_first();   // read once
      uint32_t nxt[4];
      int pt = 0, pcb = 0;                           // tile and column of the next prefetch
      auto prefetch = [&]() {
        const uint16_t* row = pcb + jl < act ? colbase[c0 + pcb + jl] : nullptr;
        load_base8(a, row, row0 + pt * 128 + 32 * q + 8 * hl, vec, base_policy, nxt);
        pcb += kCW;
        if (pcb >= cpt * kCW) { pcb = 0; ++pt; }
      };
      if (nc > 0) prefetch();
      // each chunk's scoring kind, for the whole step (columns and their
      // temperatures are fixed for the round): 2 bits per chunk
      uint32_t kinds = 0u;
      for (int cc = 0; cc < cpt; ++cc) {
        const int cj = cc * kCW + jl;
        const float Tj = cj < act ? tcol[c0 + cj] : 0.0f;
        const uint32_t kd = __any_sync(0xFFFFFFFFu, Tj > 0.0f) ? (a.sampler == 1 ? 2u : 1u) : 0u;
        kinds |= kd << (2 * cc);
      }
      int ci = 0;
      for (int t = 0; t < T; ++t) {
        const int Gt = G + t;
        const int d = Gt & 1;
        if (!wait_bar(&dfull[d], (uint32_t)((Gt >> 1) & 1), t_step, a.timeout_ns)) {
          if (lane == 0) {
            abort_round(a.sync.hdr, round_s, kStatusTimeout);
            abort_s = 1;
          }
          break;
        }
        ptx::tc_fence_after();
        if (t == 0) trace_stamp(a, k, 1);
        const int64_t v0 = row0 + t * 128 + 32 * q + 8 * hl;
        for (int cc = 0; cc < cpt; ++cc, ++ci) {
          const int cb = cc * kCW;
          uint32_t cur[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
          if (ci + 1 < nc) prefetch();
          uint32_t dv[kCW];
          ptx::tmem_ld<kCW>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * 256 + c0 + cb), dv);
          ptx::tmem_wait_ld();
          // bf16 biases, one row per lane, then read back one column per lane
          __syncwarp();
#pragma unroll
          for (int j = 0; j < kCW; ++j)
            stg[j * kStgStride + lane] = float_to_bf16_bits_rn(__uint_as_float(dv[j]));
          __syncwarp();
          const uint4 bz = *reinterpret_cast<const uint4*>(stg + jl * kStgStride + 8 * hl);
          unsigned long long best = 0ull;
          const bool live = cb + jl < act;
          const int c = c0 + cb + jl;
          const float Tc = live ? tcol[c] : 0.0f, iTc = live ? icol[c] : 1.0f;
          const int kind = (int)((kinds >> (2 * cc)) & 3u);
          if (live) best = score8(a, pk, k, (int)col2req[c], Tc, iTc, v0, bz, cur, vec, kind);
          unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, best, 8);
          best = o > best ? o : best;
          o = __shfl_xor_sync(0xFFFFFFFFu, best, 16);
          best = o > best ? o : best;
          if (hl == 0 && live) {
            unsigned long long* p = &wbest[warp * kWbCols + cb + jl];
            *p = best > *p ? best : *p;
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[d]);
      }
      trace_stamp(a, k, 2);
      G += T;
    }
    __syncthreads();
    trace_stamp(a, k, 3);
    if (abort_s) { ok = false; break; }

    // CTA best per request: max over the 4 lane quarters of its column
    for (int c = threadIdx.x; c < N; c += blockDim.x) {
      if (col2req[c] < 0) continue;
      const int grp = c / (N >> 2), j = c - grp * (N >> 2);
      unsigned long long m = 0ull;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const unsigned long long x = wbest[(grp * 4 + qq) * kWbCols + j];
        m = x > m ? x : m;
      }
      cta_key[col2req[c]] = m;
    }
    __syncthreads();
    trace_stamp(a, k, 4);
    ok = exchange(a, round_s, k, cta_key, tok_s, &flag_s);
    trace_stamp(a, k, 5);
    if (!ok) break;
    if (cta == 0)
      for (int b = threadIdx.x; b < a.B; b += blockDim.x)
        a.out_tokens[(size_t)b * a.gamma + k] = tok_s[b];
    if (k + 1 < a.gamma && warp < kEpiWarps) gather_u(a, tok_s, col2req, U, N);
    for (int c = threadIdx.x; c < 256; c += blockDim.x)     // next step's base rows
      if (colbase[c] != nullptr) colbase[c] += a.V;
    ptx::tc_fence_before();
    __syncthreads();
    trace_stamp(a, k, 7);
  }

  // ----------------------------------------------------------------- exit --
  // let every copy this CTA issued land before the CTA (and its shared
  // memory) goes away; all issued MMAs were waited for by the epilogue
  if (warp == kEpiWarps && lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (int i = consumed; i < issued; ++i)
      (void)wait_bar(&full_bar[i % nst], (uint32_t)((i / nst) & 1), t0, a.timeout_ns);
    for (int i = (consumed > nst ? consumed - nst : 0); i < consumed; ++i)
      (void)wait_bar(&empty_bar[i % nst], (uint32_t)((i / nst) & 1), t0, a.timeout_ns);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kEpiWarps) ptx::tmem_dealloc(tmem, 512);
  if (cta == 0) {
    if (!ok)
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    if (threadIdx.x == 0) atomicAdd(&a.sync.hdr->round, 1u);
  }
}

// Row-major W2 -> per CTA, per 128-row tile, per 16-wide K block a 4 KB block
// of 8x16-byte core matrices: row r = 8 mg + i, k = 8 kc + j at byte
// ((kc * 16 + mg) * 8 + i) * 16 + 2 j.  Rows past V are zero.
__global__ void repack_batched_kernel(uint32_t* __restrict__ W2w, uint32_t* __restrict__ out,
                                      int64_t V, int R, int64_t total_words, int inverse) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = i >> 10;              // 1024 words per 4 KB block
    const int w = (int)(i & 1023);
    const int jp = w & 3, ii = (w >> 2) & 7, mg = (w >> 5) & 15, kc = (w >> 9) & 1;
    const int64_t kt = blk & 15;
    const int64_t tile = blk >> 4;            // global tile index (CTA-major)
    const int64_t tiles_per_cta = R / 128;
    const int64_t cta = tile / tiles_per_cta, t = tile - cta * tiles_per_cta;
    const int64_t row = cta * R + t * 128 + 8 * mg + ii;
    const int64_t kp = kt * 8 + kc * 4 + jp;  // word (pair) index along K
    if (inverse) {
      if (row < V) W2w[row * (kRank / 2) + kp] = out[i];
    } else {
      out[i] = row < V ? W2w[row * (kRank / 2) + kp] : 0u;
    }
  }
}

}  // namespace

int batched_threads() { return kBatThreads; }

size_t batched_smem_bytes(int nst, int N) {
  return (size_t)nst * kStageBytes + (size_t)N * 512 + (size_t)kEpiWarps * kWbCols * 8 + 256 * 8 +
         256 * 4 + 256 * 4 + 256 * 2 + 256 * 4 + 256 * 4 + (size_t)kEpiWarps * kStgWarpElems * 2 +
         256 * 8;
}

int batched_max_stages() { return kMaxStages; }

const void* batched_kernel() { return reinterpret_cast<const void*>(&walk_batched_kernel); }

cudaError_t batched_repack(void* rowmajor, void* packed, int64_t V, int R, int n_cta,
                           bool inverse, cudaStream_t stream) {
  const int64_t total = (int64_t)n_cta * (R / 128) * 16 * 1024;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  repack_batched_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint32_t*>(rowmajor),
                                                    static_cast<uint32_t*>(packed), V, R, total,
                                                    inverse ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t batched_launch(const WalkArgs& w, const void* W2b, int R, int n_cta, int max_B,
                           int B, size_t smem_budget, cudaStream_t stream) {
  BatchedArgs ba{};
  ba.w = w;
  ba.W2b = static_cast<const uint8_t*>(W2b);
  ba.R = R;
  ba.T = R / 128;
  ba.N = (B + 15) / 16 * 16;
  ba.max_B = max_B;
  const size_t fixed = batched_smem_bytes(0, ba.N);
  int nst = (int)((smem_budget - fixed) / kStageBytes);
  if (nst > kMaxStages) nst = kMaxStages;
  if (nst < 2) return cudaErrorInvalidValue;
  ba.nst = nst;
  void* args[] = {&ba};
  return cudaLaunchCooperativeKernel(batched_kernel(), dim3(n_cta), dim3(kBatThreads), args,
                                     batched_smem_bytes(nst, ba.N), stream);
}

}  // namespace dspark
