// walk_common.cuh -- device pieces shared by every walk kernel: the fused
// epilogue (two bf16 roundings), the selection score (greedy or Philox
// Gumbel-max), the 64-bit selection key and the cross-CTA rendezvous.
//
// Source: "Keeping the Draft Walk on Chip: One Launch for DSpark's Markov
// Head", sections "The serial part of a parallel drafter" (recurrence, the
// bf16 rounding of W2 @ u before the add), "The idea: make the walk resident"
// (64-bit {order-preserving logit bits, inverted row index} key; {key, count}
// rendezvous with an atomic max and an atomic add; per-round state that
// alternates by round parity; Philox-keyed Gumbel-max; per-request
// temperatures read on the device) and "B200: the bf16 table fits on chip"
// (fp32 accumulation, bias rounded to bf16, sum rounded to bf16).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace dspark {

constexpr int kRank = 256;         // r: the Markov head's latent width
constexpr int kMaxB = 256;         // largest batch one round may carry
constexpr int kMaxGamma = 64;      // longest walk one round may carry

// Device-side status codes (same values as the public DSPARK_E* codes).
constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = -4;
constexpr int kStatusAnchor = -5;
constexpr int kStatusTemp = -7;
constexpr int kStatusInternal = -9;

// Rendezvous state owned by a handle, in global memory.
//   header: round counter (selects the parity) and the sticky status word;
//   count[p][k]: CTAs that have posted step k in a round of parity p
//                (one 32-byte sector each);
//   key[p][k][b]: running maximum of the posted 64-bit keys.
// A round of parity p clears parity p^1 at entry, so no memset is needed
// between rounds (or between CUDA-graph replays).
struct SyncHeader {
  uint32_t round;
  int32_t status;
  uint32_t abort_round;  // round + 1 of the last round a CTA gave up on
  uint32_t pad[5];
};
constexpr int kCountStride = 16;  // uint32 per count slot (64 bytes: one per request <= 16)

struct SyncView {
  SyncHeader* hdr;
  uint32_t* count;             // [2][max_gamma][kCountStride]
  unsigned long long* key;     // [2][max_gamma][max_B]
  int max_gamma;
  int max_B;
  // tagged slots (the mma.sync resident kernel): [2][max_gamma][slot_B][slot_stride]
  unsigned long long* slot;
  int slot_B;                  // requests with slots (min(max_B, 16))
  int slot_stride;             // words per (parity, step, request): >= CTAs, even

  __device__ __forceinline__ unsigned long long* slot_at(uint32_t parity, int k, int b) const {
    return slot + (((size_t)parity * max_gamma + k) * slot_B + b) * slot_stride;
  }

  __device__ __forceinline__ uint32_t* count_at(uint32_t parity, int k) const {
    return count + ((size_t)parity * max_gamma + k) * kCountStride;
  }
  __device__ __forceinline__ unsigned long long* key_at(uint32_t parity, int k, int b) const {
    return key + ((size_t)parity * max_gamma + k) * max_B + b;
  }
};

// Give up on the current round: record the status (first error wins) and
// mark the round, so every other CTA of THIS round stops waiting.  A status
// left over from an earlier round does not stop later rounds.
__device__ __forceinline__ void abort_round(SyncHeader* hdr, uint32_t round, int code) {
  atomicCAS(reinterpret_cast<int*>(&hdr->status), 0, code);
  atomicExch(&hdr->abort_round, round + 1u);
}

__device__ __forceinline__ bool round_aborted(const SyncHeader* hdr, uint32_t round) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(&hdr->abort_round) : "memory");
  return v == round + 1u;
}

// Everything a launch needs (passed by value).
constexpr int kCellP = 3 * kRank;   // largest recurrent product per request (the GRU's)

struct WalkArgs {
  const uint16_t* W1;          // [V, 256] bf16
  const uint16_t* W2;          // [V, 256] bf16, row-major (streamed kernels)
  const uint16_t* base;        // [B, gamma, V] bf16
  const int32_t* anchor;       // [B]
  const float* temperature;    // [B]
  int32_t* out_tokens;         // [B, gamma]
  uint16_t* out_logits;        // [B, gamma, V] bf16 or null
  SyncView sync;
  int64_t V;
  int B;
  int gamma;
  int rows_per_cta;            // shard size (last shard may be shorter)
  uint32_t seed_lo, seed_hi;   // Philox key (see round_seed)
  int seed_per_round;          // add the handle's round counter to the key
  int sampler;                 // 0: per-token Gumbel-max; 1: group inverse-CDF
  int64_t timeout_ns;          // rendezvous wait limit
  int skip_cta;                // fault injection: this CTA never posts (-1: off)
  unsigned long long* trace;   // optional [n_cta][gamma + 1][8] stamps
  int trace_global;            // stamps in global-timer ns (comparable across SMs), not SM clocks
  // recurrent heads (resident kernel only)
  int cell;                    // 0: Markov (u = W1[prev]); 1: gated; 2: RNN; 3: GRU
  const uint16_t* cell_M;      // [P, 256] bf16 recurrent rows (P = 256; GRU: 768)
  const uint16_t* cell_X;      // GRU: [3, V, 256] bf16 token tables (r, z, n)
  float* cell_p;               // [gamma][16][kCellP] fp32: M @ h_k, published slice by slice
  int cell_q;                  // rows of M per CTA: CTA c owns rows [c q, c q + q)
  uint16_t* out_state;         // [B, gamma, 256] bf16 states u_k, or null
};


__device__ __forceinline__ uint64_t globaltimer_ns();

// Phase stamp of thread 0 into the optional trace buffer (SM clock cycles, or
// global-timer nanoseconds, which compare across SMs): slot k < gamma is step
// k, slot gamma is the round's entry.
__device__ __forceinline__ void trace_stamp(const WalkArgs& a, int slot, int phase) {
  if (a.trace != nullptr && threadIdx.x == 0)
    a.trace[((size_t)blockIdx.x * (a.gamma + 1) + slot) * 8 + phase] =
        a.trace_global ? globaltimer_ns() : (unsigned long long)clock64();
}

// The Philox key of this round: the seed, plus the round counter when the
// handle keys its noise per round (seed + n mod 2^64), as two 32-bit words.
__device__ __forceinline__ uint2 round_seed(const WalkArgs& a, uint32_t round) {
  uint64_t s = ((uint64_t)a.seed_hi << 32) | a.seed_lo;
  if (a.seed_per_round) s += round;
  return make_uint2((uint32_t)s, (uint32_t)(s >> 32));
}

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float ld_relaxed_gpu_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ld_relaxed_gpu_s32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_relaxed_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_relaxed_gpu_max_u64(unsigned long long* p,
                                                        unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void set_status(SyncHeader* hdr, int code) {
  atomicCAS(reinterpret_cast<int*>(&hdr->status), 0, code);
}

// ------------------------------------------------------------------ bf16 --

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) {
  return __uint_as_float(h << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// One element of a recurrent head's state update ("Keeping the Draft Walk on
// Chip", section "Beyond DSpark: other serial heads"; the pages print no cell
// equations, these are the plain gated and Elman forms): from p = M[i, :] .
// h_{k-1}, the token's W1 element x and the previous state element hp,
//   gated: z = 1 / (1 + exp(-p)), (1 - z) hp + z x;   RNN: tanh(p + x);
// in fp32, each operation rounded (no contraction), then rounded to bf16.
__device__ __forceinline__ uint16_t cell_element(int cell, float p, float x, float hp) {
  float v;
  if (cell == 1) {
    const float z = __frcp_rn(__fadd_rn(1.0f, expf(-p)));
    v = __fadd_rn(__fmul_rn(__fsub_rn(1.0f, z), hp), __fmul_rn(z, x));
  } else {
    v = tanhf(__fadd_rn(p, x));
  }
  return float_to_bf16_bits_rn(v);
}

// One element of the GRU head's update (the same page; the usual reset /
// update gate form, input projections folded into the token tables): from
// the recurrent products pr, pz, pn, the token's table elements xr, xz, xn and
// the previous state element hp, r = sig(xr + pr), z = sig(xz + pz),
// n = tanh(xn + r pn), (1 - z) n + z hp; fp32, each operation rounded.
__device__ __forceinline__ uint16_t gru_element(float pr, float pz, float pn, float xr, float xz,
                                                float xn, float hp) {
  const float r = __frcp_rn(__fadd_rn(1.0f, expf(-__fadd_rn(xr, pr))));
  const float z = __frcp_rn(__fadd_rn(1.0f, expf(-__fadd_rn(xz, pz))));
  const float n = tanhf(__fadd_rn(xn, __fmul_rn(r, pn)));
  return float_to_bf16_bits_rn(__fadd_rn(__fmul_rn(__fsub_rn(1.0f, z), n), __fmul_rn(z, hp)));
}

// ------------------------------------------------------------------- key --

// Order-preserving map of an fp32 value to 32 bits (larger value, larger
// bits); -0 is folded onto +0 so that the two compare equal.
__device__ __forceinline__ uint32_t ord32(float x) {
  if (x == 0.0f) x = 0.0f;
  uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// {score bits : 32, inverted token id : 32}: the maximum key is the largest
// score, and among equal scores the smallest token id.  Key 0 is below every
// real key (ord32 of -inf is 0x007FFFFF), so a zeroed slot means "empty".
__device__ __forceinline__ unsigned long long make_key(float s, uint32_t v) {
  return ((unsigned long long)ord32(s) << 32) | (unsigned long long)(0xFFFFFFFFu - v);
}

__device__ __forceinline__ int32_t key_token(unsigned long long key) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)key);
}

// ---------------------------------------------------------------- Philox --

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies; round i uses the key bumped i times by the Weyl
// constants.  The round keys depend on the seed alone, so a thread that draws
// many blocks computes them once.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys p;
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    p.k0[i] = k0 + (uint32_t)i * 0x9E3779B9u;
    p.k1[i] = k1 + (uint32_t)i * 0xBB67AE85u;
  }
  return p;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& key) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ key.k0[i], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ key.k1[i], (uint32_t)p0);
  }
  return c;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  return philox4x32_10(c, philox_keys(k0, k1));
}

__device__ __forceinline__ uint32_t philox_word(uint4 r, uint32_t w) {
  return w == 0 ? r.x : (w == 1 ? r.y : (w == 2 ? r.z : r.w));
}

// Random bits -> fp32 uniform: the midpoint of bin (x >> 9) of 2^23 bins,
// exact in fp32 and strictly inside (0, 1): (2 (x >> 9) + 1) 2^-24, formed as
// 1.m - (1 - 2^-24) with m = x >> 9 in the mantissa of 1.0 (the subtraction
// is exact by Sterbenz's lemma), so no int -> float conversion (a quarter-rate
// instruction) is spent per token.
__device__ __forceinline__ float bits_to_uniform(uint32_t x) {
  return __fsub_rn(__uint_as_float(0x3F800000u | (x >> 9)), 0x1.fffffep-1f);
}

// log2 by the hardware approximation, subnormal inputs flushed (the noise
// never feeds it one: U >= 2^-24 and -log U >= 2^-24).
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// -log U for the uniform of bits x.  For U <= 15/16 the hardware log2
// approximation times ln 2: its absolute error (about 2^-22 in log2 near 1,
// relative elsewhere) is then below 2^-18 of -log U >= 0.0645.  For U > 15/16,
// t = 1 - U is exact and -log(1 - t) = t + t^2/2 + ... + t^6/6 (the Mercator
// series, remainder below t^7 / 7 < 2^-28 t), so the tokens whose U is close
// to 1 -- the large-noise ones that tend to win -- keep full precision.
__device__ __forceinline__ float neg_log_uniform(uint32_t x) {
  const float U = bits_to_uniform(x);
  const float t = 1.0f - U;
  float p = fmaf(t, 1.0f / 6.0f, 0.2f);
  p = fmaf(t, p, 0.25f);
  p = fmaf(t, p, 1.0f / 3.0f);
  p = fmaf(t, p, 0.5f);
  p = fmaf(t, p, 1.0f);
  const float series = t * p;
  const float hw = -0.693147180559945f * lg2_approx(U);
  return t < 0.0625f ? series : hw;
}

// Gumbel noise g = -log(-log U): the inner log as above, the outer one the
// hardware approximation (absolute error below 2^-21 for arguments in
// [0.5, 2], a few ulp elsewhere).  Both stay far inside the 2^-18 (1 + |g|)
// error the token comparison allows for the noise.
__device__ __forceinline__ float gumbel_noise(uint32_t x) {
  return -0.693147180559945f * lg2_approx(neg_log_uniform(x));
}

// Gumbel-max score of a logit at temperature T > 0: fp32(logit / T) + g, in
// fp32.  inv_T = fl(1/T) (0 when 1/T overflows): the quotient is taken as the
// product with the rounded reciprocal, within one fp32 ulp of the IEEE
// quotient.
__device__ __forceinline__ float gumbel_score(float logit, float T, float inv_T, uint32_t x) {
  const float q = inv_T != 0.0f ? __fmul_rn(logit, inv_T) : __fdiv_rn(logit, T);
  return __fadd_rn(q, gumbel_noise(x));
}

// exp2 by the hardware approximation, subnormal results flushed.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Group inverse-CDF sampling ("Keeping the Draft Walk on Chip...", section
// "The idea: make the walk resident": an inverse CDF inside 8-row groups and
// Gumbel-max across them; vLLM pull request #64442, section "Details": a
// uniform times the mass picks the first token whose running sum of fp32
// weights passes it).  For the group j of tokens v0 = 8j .. v0 + n - 1 of
// request b at step k, with fp32 logits lg: z = logit / T (product with
// fl(1/T) unless that overflows), m = max z, weights w = exp(z - m), mass S;
// score = m + log S - log(-log U1); pick = the first token whose running sum
// of weights exceeds U2 * S (the last one if rounding leaves none).  U1, U2 are
// the words 2 (j & 1) and 2 (j & 1) + 1 of Philox counter (j >> 1, k, b, 1).
// Returns the group's selection key {ord32(score), inverted id of the pick}.
// kQ: how fp32(logit / T) is formed -- 0: the product with inv_T; 1: the IEEE
// quotient; 2: the product, or the quotient where inv_T is 0, per element.
template <int kQ>
__device__ __forceinline__ unsigned long long group_key_q(const float (&lg)[8], int n, float T,
                                                          float inv_T, uint32_t v0, int k, int b,
                                                          const PhiloxKeys& pk) {
  float z[8];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q = kQ == 0   ? __fmul_rn(lg[i], inv_T)
                    : kQ == 1 ? __fdiv_rn(lg[i], T)
                              : (inv_T != 0.0f ? __fmul_rn(lg[i], inv_T) : __fdiv_rn(lg[i], T));
    z[i] = i < n ? q : -INFINITY;
    m = fmaxf(m, z[i]);
  }
  float w[8];
  float S = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w[i] = i < n ? ex2_approx(__fmul_rn(__fsub_rn(z[i], m), 1.4426950408889634f)) : 0.0f;
    S = __fadd_rn(S, w[i]);
  }
  const uint32_t j = v0 >> 3;
  const uint4 r = philox4x32_10(make_uint4(j >> 1, (uint32_t)k, (uint32_t)b, 1u), pk);
  const uint32_t x1 = (j & 1u) ? r.z : r.x;
  const uint32_t x2 = (j & 1u) ? r.w : r.y;
  const float score =
      __fadd_rn(__fadd_rn(m, 0.693147180559945f * lg2_approx(S)), gumbel_noise(x1));
  const float target = __fmul_rn(bits_to_uniform(x2), S);
  float run = 0.0f;
  int pick = n - 1;
  float runs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    run = __fadd_rn(run, w[i]);
    runs[i] = run;
  }
#pragma unroll
  for (int i = 7; i >= 0; --i)
    if (i < n && runs[i] > target) pick = i;
  return ((unsigned long long)ord32(score) << 32) |
         (unsigned long long)(0xFFFFFFFFu - (v0 + (uint32_t)pick));
}

// The group key with the IEEE quotient, for a temperature whose reciprocal
// overflows (T below 2^-126).  Out of line, arguments by value: the rare form
// costs the common one neither registers nor instructions.
static __device__ __noinline__ unsigned long long group_key_div(
    float l0, float l1, float l2, float l3, float l4, float l5, float l6, float l7, int n,
    float T, uint32_t v0, int k, int b, uint32_t key0, uint32_t key1) {
  const float lg[8] = {l0, l1, l2, l3, l4, l5, l6, l7};
  return group_key_q<1>(lg, n, T, 0.0f, v0, k, b, philox_keys(key0, key1));
}

// The group key of tokens v0 .. v0 + n - 1 (see group_key_q); inv_T = fl(1/T),
// 0 when that overflows.
__device__ __forceinline__ unsigned long long group_key(const float (&lg)[8], int n, float T,
                                                        float inv_T, uint32_t v0, int k, int b,
                                                        const PhiloxKeys& pk) {
  if (inv_T == 0.0f)
    return group_key_div(lg[0], lg[1], lg[2], lg[3], lg[4], lg[5], lg[6], lg[7], n, T, v0, k, b,
                         pk.k0[0], pk.k1[0]);
  return group_key_q<0>(lg, n, T, inv_T, v0, k, b, pk);
}

// fl(1/T) for T > 0, or 0 when it overflows (T below 2^-126).
__device__ __forceinline__ float inv_temperature(float T) {
  const float r = __frcp_rn(T);
  return isinf(r) ? 0.0f : r;
}

// ------------------------------------------------------------- epilogue --

// Gumbel-max score of token v (request b, step k) at temperature T > 0.  Kept
// out of line: the walk kernels inline the epilogue at many sites, and ten
// Philox rounds plus two logs at each of them would overflow the instruction
// cache on the (common) greedy path.
static __device__ __noinline__ float sampled_score(float logit, float T, uint32_t seed_lo,
                                            uint32_t seed_hi, int b, int k, uint32_t v) {
  const uint4 r = philox4x32_10(make_uint4(v >> 2, (uint32_t)k, (uint32_t)b, 0u), seed_lo,
                                seed_hi);
  return gumbel_score(logit, T, inv_temperature(T), philox_word(r, v & 3u));
}

// The fused epilogue of one (token v, request b, step k): fp32 accumulation
// -> bf16 bias; fp32 add of the base logit -> bf16 logit; selection score.
// Returns the selection key; *logit_bits receives the bf16 logit.
__device__ __forceinline__ unsigned long long epilogue_key(
    float acc, uint32_t base_bits, float T, uint32_t seed_lo, uint32_t seed_hi, int b, int k,
    uint32_t v, uint16_t* logit_bits) {
  const float bias = __bfloat162float(__float2bfloat16_rn(acc));
  const uint16_t lb = float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(base_bits), bias));
  *logit_bits = lb;
  const float logit = bf16_bits_to_float(lb);
  float s = logit;
  if (T > 0.0f) s = sampled_score(logit, T, seed_lo, seed_hi, b, k, v);
  return make_key(s, v);
}

// ----------------------------------------------------------- rendezvous --

// Entry checks every CTA makes on its own (so all agree without talking):
// anchors inside [0, V), temperatures finite and >= 0.  Returns the status.
__device__ __forceinline__ int check_inputs(const WalkArgs& a, int* flag_smem) {
  if (threadIdx.x == 0) *flag_smem = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int32_t an = a.anchor[b];
    const float T = a.temperature[b];
    if (an < 0 || (int64_t)an >= a.V) atomicCAS(flag_smem, 0, kStatusAnchor);
    if (!(T >= 0.0f) || isinf(T)) atomicCAS(flag_smem, 0, kStatusTemp);
  }
  __syncthreads();
  return *flag_smem;
}

// Clear the rendezvous slots of the other parity (CTA 0 only).
__device__ __forceinline__ void clear_other_parity(const SyncView& s, uint32_t parity) {
  const uint32_t q = parity ^ 1u;
  uint32_t* c = s.count_at(q, 0);
  for (int i = threadIdx.x; i < s.max_gamma * kCountStride; i += blockDim.x) c[i] = 0u;
  unsigned long long* kk = s.key_at(q, 0, 0);
  for (int i = threadIdx.x; i < s.max_gamma * s.max_B; i += blockDim.x) kk[i] = 0ull;
}

// Tagged-slot exchange: CTA c's best key of request b at step k of a round is
// one 64-bit word slot_at(parity, k, b)[c] = {round tag : 14, key : 50}.  The
// tag makes the word self-validating, so the post is one relaxed store with no
// fence and no atomic; a reader polls all CTAs' words until each carries this
// round's tag.  Every CTA clears its own words of the other parity at entry, so
// the next round never sees a stale word of the same tag.
__device__ __forceinline__ unsigned long long slot_tag(uint32_t round) {
  return (unsigned long long)((round & 0x1FFFu) | 0x2000u) << 50;
}

// The 64-bit key {order bits : 32, 0xFFFFFFFF - v} packed into 50 bits
// {order bits : 32, 0x3FFFF - v} (same order for token ids v < 2^18).
__device__ __forceinline__ unsigned long long key50(unsigned long long key64) {
  return ((key64 >> 32) << 18) | (key64 & 0x3FFFFull);
}

__device__ __forceinline__ int32_t key50_token(unsigned long long k) {
  return (int32_t)(0x3FFFFu - (uint32_t)(k & 0x3FFFFull));
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void ld_relaxed_gpu_v2u64(const unsigned long long* p,
                                                     unsigned long long& a,
                                                     unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// This CTA's words of the other parity, zeroed (all threads of the CTA).
__device__ __forceinline__ void clear_own_slots(const SyncView& s, uint32_t parity) {
  const uint32_t q = parity ^ 1u;
  for (int i = threadIdx.x; i < s.max_gamma * s.slot_B; i += blockDim.x)
    s.slot_at(q, i / s.slot_B, i % s.slot_B)[blockIdx.x] = 0ull;
}

// One step's cross-CTA selection.  cta_key[b] holds this CTA's best key of
// request b; on return tok_smem[b] holds the common winner of request b.
// Returns false if the wait ran out or another CTA reported an error; then
// every CTA leaves the walk.
__device__ __forceinline__ bool exchange(const WalkArgs& a, uint32_t round, int k,
                                         const unsigned long long* cta_key, int32_t* tok_smem,
                                         int* flag_smem) {
  const uint32_t parity = round & 1u;
  const bool post = (int)blockIdx.x != a.skip_cta;
  if (post) {
    for (int b = threadIdx.x; b < a.B; b += blockDim.x)
      red_relaxed_gpu_max_u64(a.sync.key_at(parity, k, b), cta_key[b]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    uint32_t* cnt = a.sync.count_at(parity, k);
    // the release is cumulative over the maxima the CTA barrier ordered
    // before it (no separate fence)
    if (post) red_release_gpu_add(cnt, 1u);
    const uint32_t target = gridDim.x;
    const uint64_t t0 = globaltimer_ns();
    uint32_t spins = 0;
    while (ld_acquire_gpu(cnt) < target) {
      if ((++spins & 63u) == 0u) {
        if (round_aborted(a.sync.hdr, round)) { ok = 0; break; }
        if ((int64_t)(globaltimer_ns() - t0) > a.timeout_ns) {
          abort_round(a.sync.hdr, round, kStatusTimeout);
          ok = 0;
          break;
        }
      }
    }
    *flag_smem = ok;
  }
  __syncthreads();
  const bool ok = *flag_smem != 0;
  if (ok) {
    for (int b = threadIdx.x; b < a.B; b += blockDim.x)
      tok_smem[b] = key_token(ld_acquire_gpu_u64(a.sync.key_at(parity, k, b)));
  }
  __syncthreads();
  return ok;
}

// Arguments of the resident kernel: the common ones plus the tiered layout.
struct ResidentArgs {
  WalkArgs w;
  const uint32_t* W2p;            // repacked W2, words_per_cta words per CTA
  int R;                          // rows per CTA (multiple of 16)
  int S;                          // shared-memory strips per CTA
  int ST;                         // strips streamed every step (0: fully resident)
  int nslot;                      // ring slots (64 KB each) of the streamed strips
  int64_t words_per_cta;
  int base_mode;                  // 16, 4 or 2: bytes per base-prefetch copy
};

}  // namespace dspark
