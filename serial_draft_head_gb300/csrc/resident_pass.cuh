// resident_pass.cuh -- device pieces shared by the two resident walk kernels
// (walk_resident.cu: tcgen05.mma on the tensor-memory tier; walk_mma_resident.cu:
// every tier through mma.sync): the base-logit prefetch, the gather of the
// next latents u = W1[prev], the recurrent heads' exchange rows, the in-place
// logits of an mma.sync strip, and the key pass that scores every logit of a
// CTA's shard ("Keeping the Draft Walk on Chip: One Launch for DSpark's Markov
// Head", section "The idea: make the walk resident": one CTA per SM, the
// 64-bit {order bits, inverted id} key, Philox-keyed Gumbel-max; section "B200:
// the bf16 table fits on chip": fp32 accumulation, bias rounded to bf16, then
// the sum rounded to bf16).
#pragma once

#include "tc_ptx.cuh"
#include "walk_common.cuh"

namespace dspark {
namespace {

constexpr int kResThreads = 256;
constexpr int kResWarps = kResThreads / 32;
constexpr int kSmemStripBytes = 16 * 512;

__device__ __forceinline__ unsigned long long key_max(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Maximum of a 64-bit key over the warp with two 32-bit redux.sync reductions
// (high word, then the low word among the lanes holding the high maximum).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long key) {
  const uint32_t hi = (uint32_t)(key >> 32);
  const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
  const uint32_t lo = hi == mhi ? (uint32_t)key : 0u;
  const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, lo);
  return ((unsigned long long)mhi << 32) | mlo;
}

__device__ __forceinline__ bool wait_mbar(uint64_t* bar, uint32_t parity, uint64_t t0,
                                          int64_t limit_ns) {
  uint32_t spins = 0;
  while (!ptx::mbar_try_wait(bar, parity)) {
    if ((++spins & 255u) == 0u && (int64_t)(globaltimer_ns() - t0) > limit_ns) return false;
  }
  return true;
}

// Stage base[b, k, row0 .. row0 + nv) for every request into base_s[b][0..R).
__device__ __forceinline__ void prefetch_base(const ResidentArgs& ra, int k, int64_t row0,
                                              int nv, uint16_t* base_s, int first = 0,
                                              int count = 0) {
  const WalkArgs& a = ra.w;
  if (k >= a.gamma) return;
  const int tid = (int)threadIdx.x - first;      // this thread's index among `count`
  const int nthr = count > 0 ? count : (int)blockDim.x;
  if (ra.base_mode == 16) {
    // read once: evict-first, so that the base logits do not push out W2
    // rows that a streamed tier re-reads every step
    const uint64_t pol = ptx::policy_evict_first();
    const int per = nv >> 3;
    for (int i = tid; i < a.B * per; i += nthr) {
      const int b = i / per, c = i - b * per;
      const uint16_t* src = a.base + ((size_t)b * a.gamma + k) * (size_t)a.V + row0 + 8 * c;
      ptx::cp_async16_hint(base_s + (size_t)b * ra.R + 8 * c, src, pol);
    }
  } else if (ra.base_mode == 4) {
    const int per = nv >> 1;
    for (int i = tid; i < a.B * per; i += nthr) {
      const int b = i / per, c = i - b * per;
      const uint16_t* src = a.base + ((size_t)b * a.gamma + k) * (size_t)a.V + row0 + 2 * c;
      ptx::cp_async4(base_s + (size_t)b * ra.R + 2 * c, src);
    }
  } else {
    for (int i = tid; i < a.B * nv; i += nthr) {
      const int b = i / nv, c = i - b * nv;
      base_s[(size_t)b * ra.R + c] = a.base[((size_t)b * a.gamma + k) * (size_t)a.V + row0 + c];
    }
  }
}

// u_b = W1[tok] into U (core matrix (kc, b/8), row b%8): one 16-byte chunk per lane.
// A recurrent head's first state h_0 (from h_{-1} = 0: p = 0, previous state 0)
// is formed from that row (the GRU: from the token's rows of its three tables)
// in place.
__device__ __forceinline__ void gather_u_row(const WalkArgs& a, int32_t tok, int b, uint8_t* U,
                                             int lane, int cell) {
  uint4 x = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok * kRank) + lane);
  if (cell == 3) {
    const uint4* X = reinterpret_cast<const uint4*>(a.cell_X);
    const uint4 xr = __ldg(X + ((size_t)tok) * 32 + lane);
    const uint4 xz = __ldg(X + ((size_t)a.V + tok) * 32 + lane);
    const uint4 xn = __ldg(X + ((size_t)2 * a.V + tok) * 32 + lane);
    const uint32_t rw[4] = {xr.x, xr.y, xr.z, xr.w}, zw[4] = {xz.x, xz.y, xz.z, xz.w};
    const uint32_t nw[4] = {xn.x, xn.y, xn.z, xn.w};
    uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = gru_element(0.f, 0.f, 0.f, bf16_bits_to_float(rw[j] & 0xFFFFu),
                                      bf16_bits_to_float(zw[j] & 0xFFFFu),
                                      bf16_bits_to_float(nw[j] & 0xFFFFu), 0.f);
      const uint32_t hi = gru_element(0.f, 0.f, 0.f, bf16_bits_to_float(rw[j] >> 16),
                                      bf16_bits_to_float(zw[j] >> 16),
                                      bf16_bits_to_float(nw[j] >> 16), 0.f);
      w[j] = lo | (hi << 16);
    }
  } else if (cell != 0) {
    uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = cell_element(cell, 0.0f, bf16_bits_to_float(w[j] & 0xFFFFu), 0.0f);
      const uint32_t hi = cell_element(cell, 0.0f, bf16_bits_to_float(w[j] >> 16), 0.0f);
      w[j] = lo | (hi << 16);
    }
  }
  *reinterpret_cast<uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16) = x;
  ptx::fence_proxy_async_smem();
}

// U element (i, b): the bf16 at row i of request b's column.
__device__ __forceinline__ uint16_t* u_elem(uint8_t* U, int i, int b) {
  return reinterpret_cast<uint16_t*>(U + ((i >> 3) * 2 + (b >> 3)) * 128 + (b & 7) * 16) + (i & 7);
}

// Lane l's share of sum_j m_j h_j over one row: elements 8l .. 8l + 7 (two
// bf16 per word, exact products), summed in order; a 5-level butterfly over
// the lanes then completes it (13 fp32 additions deep in all).
__device__ __forceinline__ float lane_dot(const uint4 m, const uint4 h) {
  const uint32_t mw[4] = {m.x, m.y, m.z, m.w}, hw[4] = {h.x, h.y, h.z, h.w};
  float acc = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    acc = __fmaf_rn(bf16_bits_to_float(mw[e] & 0xFFFFu), bf16_bits_to_float(hw[e] & 0xFFFFu), acc);
    acc = __fmaf_rn(bf16_bits_to_float(mw[e] >> 16), bf16_bits_to_float(hw[e] >> 16), acc);
  }
  return acc;
}

__device__ __forceinline__ float row_dot(const uint4 m, const uint4 h) {
  float acc = lane_dot(m, h);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, o));
  return acc;
}

// A recurrent head's exchange, published with this step's arrival: this CTA's
// rows of p = M @ h_k for every request (M rows [cta q, cta q + q)).  With
// q <= 8 each warp keeps one row in registers for the whole walk (`mreg`,
// row cta q + warp % q) and takes every (8 / q)-th request; otherwise (tiny
// vocabularies on few CTAs) one warp per (row, request), rows read from L2.
__device__ __forceinline__ void publish_cell_rows(const WalkArgs& a, const uint8_t* U, int k,
                                                  int cta, int warp, int lane, const uint4 mreg) {
  const int q = a.cell_q, r0 = cta * q, P = a.cell == 3 ? kCellP : kRank;
  auto u_chunk = [&](int b) {
    return *reinterpret_cast<const uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16);
  };
  if (q <= kResWarps) {
    const int j = warp % q, g = warp / q, G = kResWarps / q;
    if (g >= G || r0 + j >= P) return;
    if (a.B <= G) {                                 // one request per warp at most
      if (g < a.B) {
        const float acc = row_dot(mreg, u_chunk(g));
        if (lane == 0) a.cell_p[((size_t)k * 16 + g) * kCellP + r0 + j] = acc;
      }
      return;
    }
    for (int b0 = g; b0 < a.B; b0 += 4 * G) {      // four requests' butterflies interleaved
      float acc[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int b = b0 + t * G;
        acc[t] = b < a.B ? lane_dot(mreg, u_chunk(b)) : 0.0f;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xFFFFFFFFu, acc[t], o));
      if (lane == 0)
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int b = b0 + t * G;
          if (b < a.B) a.cell_p[((size_t)k * 16 + b) * kCellP + r0 + j] = acc[t];
        }
    }
    return;
  }
  const int nr = P - r0 < q ? P - r0 : q;
  for (int pr = warp; pr < nr * a.B; pr += kResWarps) {
    const int row = r0 + pr / a.B, b = pr % a.B;
    const uint4 m = __ldg(reinterpret_cast<const uint4*>(a.cell_M + (size_t)row * kRank) + lane);
    const float acc = row_dot(m, u_chunk(b));
    if (lane == 0) a.cell_p[((size_t)k * 16 + b) * kCellP + row] = acc;
  }
}


// In-place first half of the fused epilogue: base_s[b][rl] (the bf16 base
// logit) becomes bf16(base + bf16(acc)), the logit the token is chosen from,
// here for one 16-row strip held as mma.sync accumulators (column n = request
// n).  All base values are loaded before any logit is stored: the stores
// could otherwise alias later loads and serialise the chain.
template <int NT>
__device__ __forceinline__ void logits_strip(const float (&acc)[NT][4], uint16_t* base_s, int R,
                                             int B, int rl0, int lane) {
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t bv[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int b = 8 * nt + 2 * t4 + e;
      const bool on = b < B;
      bv[nt][e] = on ? base_s[(size_t)b * R + rl0 + g] : 0u;
      bv[nt][2 + e] = on ? base_s[(size_t)b * R + rl0 + g + 8] : 0u;
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int b = 8 * nt + 2 * t4 + e;
      if (b < B) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float bias = __bfloat162float(__float2bfloat16_rn(acc[nt][2 * h + e]));
          base_s[(size_t)b * R + rl0 + g + 8 * h] =
              float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(bv[nt][2 * h + e]), bias));
        }
      }
    }
}

// Sampled keys of request b's rows handled by this thread (blocks of 4
// tokens c = gi, gi + tpr, ...; two blocks per iteration, so two independent
// Philox chains): the best key {ord32(score), inverted id}.  FASTQ: the
// quotient logit / T as the product with fl(1/T) (else the IEEE quotient,
// when 1/T overflows).
// kTrack: keep the best score and its row in fp32 / int registers (this
// thread's rows come in increasing order, so a strict > keeps the smallest id
// among equal scores) and form the 64-bit key once, instead of a key and a
// 64-bit maximum per row.
template <bool FASTQ, bool kTrack = false>
__device__ __forceinline__ unsigned long long sampled_block_keys(
    const WalkArgs& a, const uint16_t* ls, int nv, int64_t row0, int k, int b, int gi, int tpr,
    float T, float inv_T, const PhiloxKeys& pk, uint16_t* outl) {
  unsigned long long best = 0ull;
  float bs = 0.0f;
  int bv = -1;
  for (int c = gi; 4 * c < nv; c += 2 * tpr) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int rl0 = 4 * (c + u * tpr);
      if (rl0 < nv) {
        const uint2 w = *reinterpret_cast<const uint2*>(ls + rl0);
        const uint32_t lb[4] = {w.x & 0xFFFFu, w.x >> 16, w.y & 0xFFFFu, w.y >> 16};
        const uint32_t v0 = (uint32_t)(row0 + rl0);     // a multiple of 4
        const uint4 r = philox4x32_10(make_uint4(v0 >> 2, (uint32_t)k, (uint32_t)b, 0u), pk);
        const uint32_t x[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (rl0 + e < nv) {
            const float lgt = bf16_bits_to_float(lb[e]);
            const float q = FASTQ ? __fmul_rn(lgt, inv_T) : __fdiv_rn(lgt, T);
            const float sc = __fadd_rn(q, gumbel_noise(x[e]));
            if (kTrack) {
              if (bv < 0 || sc > bs) {
                bs = sc;
                bv = (int)(v0 + e);
              }
            } else {
              const unsigned long long key = make_key(sc, v0 + e);
              best = key > best ? key : best;
            }
            if (outl) outl[v0 + e] = (uint16_t)lb[e];
          }
        }
      }
    }
  }
  if (kTrack && bv >= 0) best = make_key(bs, (uint32_t)bv);
  return best;
}

// The group sampler's keys of this thread's groups of 8 rows (see group_key_q
// for kQ), and the optional copy of the logits.
template <int kQ>
__device__ __forceinline__ unsigned long long group_block_keys(
    const uint16_t* ls, int nv, int64_t row0, int k, int b, int gi, int tpr, float T,
    float inv_T, const PhiloxKeys& pk, uint16_t* outl) {
  unsigned long long best = 0ull;
  for (int c = gi; 8 * c < nv; c += tpr) {
    const int rl0 = 8 * c;
    const uint4 w = *reinterpret_cast<const uint4*>(ls + rl0);
    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
    float lg[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      lg[e] = bf16_bits_to_float((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
    const int n = nv - rl0 < 8 ? nv - rl0 : 8;
    const uint32_t v0 = (uint32_t)(row0 + rl0);     // a multiple of 8
    const unsigned long long key = group_key_q<kQ>(lg, n, T, inv_T, v0, k, b, pk);
    best = key > best ? key : best;
    if (outl)
      for (int e = 0; e < n; ++e) outl[v0 + e] = (uint16_t)((wd[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
  }
  return best;
}

// Second half, over all of the CTA's rows: selection score and key of each
// logit (greedy: the logit; sampled: Philox Gumbel-max, one Philox call per 4
// consecutive tokens), the best key per (request, thread group), and the
// optional copy of the logits for the verifier.  Requests run side by side:
// `tpr` = blockDim / (B rounded up to a power of two) threads per request.
// group_best[b][slot] receives one key per group of 32 (or 16) threads.
struct KeyPassMap {      // this thread's share of the key pass (fixed for a round)
  int tpr;              // threads per request: blockDim / (B rounded up to a power of 2)
  int b, gi;            // request, index among its tpr threads
  float T, inv_T;       // the request's temperature and fl(1/T)
};

__device__ __forceinline__ KeyPassMap key_pass_map(int B, const float* temp_s) {
  int bp = 1;
  while (bp < B) bp <<= 1;
  KeyPassMap m;
  m.tpr = kResThreads / bp;                        // 16 .. 256
  m.b = (int)threadIdx.x / m.tpr;
  m.gi = (int)threadIdx.x % m.tpr;
  m.T = m.b < B ? temp_s[m.b] : 0.0f;
  m.inv_T = m.T > 0.0f ? inv_temperature(m.T) : 0.0f;
  return m;
}

// kHoistQ (the B > 8 instantiations): the group sampler picks its quotient
// form once per thread instead of per element (8% faster at B=16), and the
// Gumbel rows track their best in fp32 (sampled_block_keys' kTrack).  The
// B <= 8 instantiations keep the older code, with which the fully resident k
// loop runs 0.35 us faster per round.
template <bool kHoistQ>
__device__ __forceinline__ void key_pass(const WalkArgs& a, const uint16_t* logit_s, int R,
                                         int nv, int64_t row0, int k, const KeyPassMap& m,
                                         uint2 seed,
                                         unsigned long long (*group_best)[kResWarps]) {
  const int tpr = m.tpr, b = m.b, gi = m.gi;
  const int lane = threadIdx.x & 31;
  unsigned long long best = 0ull;
  if (b < a.B) {
    const float T = m.T;
    const float inv_T = m.inv_T;
    const uint16_t* ls = logit_s + (size_t)b * R;
    uint16_t* outl =
        a.out_logits ? a.out_logits + ((size_t)b * a.gamma + k) * (size_t)a.V : nullptr;
    // separate loops: one loop with a select would evaluate the noise always
    if (T > 0.0f && a.sampler == 1) {
      // group sampler: one group of 8 rows (16 bytes of logits) per iteration;
      // the quotient's form chosen once, outside the loop
      const PhiloxKeys pk = philox_keys(seed.x, seed.y);
      if (!kHoistQ)
        best = group_block_keys<2>(ls, nv, row0, k, b, gi, tpr, T, inv_T, pk, outl);
      else
        best = inv_T != 0.0f
                   ? group_block_keys<0>(ls, nv, row0, k, b, gi, tpr, T, inv_T, pk, outl)
                   : group_block_keys<1>(ls, nv, row0, k, b, gi, tpr, T, inv_T, pk, outl);
    } else if (T > 0.0f) {
      const PhiloxKeys pk = philox_keys(seed.x, seed.y);
      // the quotient by the rounded reciprocal unless 1/T overflows
      best = inv_T != 0.0f ? sampled_block_keys<true, kHoistQ>(a, ls, nv, row0, k, b, gi, tpr, T,
                                                                inv_T, pk, outl)
                           : sampled_block_keys<false, kHoistQ>(a, ls, nv, row0, k, b, gi, tpr, T,
                                                                 inv_T, pk, outl);
    } else {
      // 32-bit keys {order bits of the bf16 logit : 16, inverted local row :
      // 16}, 8 rows per 16-byte load, two rows per 32-bit word (the order map
      // and -0 -> +0 on both halves at once), four independent maxima per
      // thread, widened to the 64-bit key once
      uint32_t mx[4] = {0u, 0u, 0u, 0u};
      for (int c = gi; 8 * c < nv; c += tpr) {
        const int rl0 = 8 * c;
        const uint4 w = *reinterpret_cast<const uint4*>(ls + rl0);
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          uint32_t x = wd[p];
          x &= ~(__vcmpeq2(x, 0x80008000u) & 0x80008000u);           // -0 -> +0
          const uint32_t sg = x & 0x80008000u;
          const uint32_t o = x ^ (sg | ((sg >> 15) * 0x7FFFu) | 0x80008000u);   // order bits
          const uint32_t r = (uint32_t)(rl0 + 2 * p);
          const uint32_t k0 = (int)r < nv ? (o << 16) | (0xFFFFu - r) : 0u;
          const uint32_t k1 = (int)r + 1 < nv ? (o & 0xFFFF0000u) | (0xFFFEu - r) : 0u;
          mx[p] = max(mx[p], max(k0, k1));
        }
        if (outl)
          for (int e = 0; e < 8 && rl0 + e < nv; ++e)
            outl[row0 + rl0 + e] = (uint16_t)(wd[e >> 1] >> (16 * (e & 1)));
      }
      const uint32_t m = max(max(mx[0], mx[1]), max(mx[2], mx[3]));
      if (m != 0u) {
        const uint32_t v = (uint32_t)(row0 + (0xFFFFu - (m & 0xFFFFu)));
        best = ((unsigned long long)(m >> 16) << 32) | (unsigned long long)(0xFFFFFFFFu - v);
      }
    }
  }
  if (tpr >= 32) {                                 // whole warps per request
    best = warp_max_key(best);
    if (lane == 0 && b < a.B) group_best[b][(threadIdx.x % tpr) >> 5] = best;
  } else {                                         // two requests per warp
    const unsigned mask = 0xFFFFu << (lane & 16);
    const uint32_t hi = (uint32_t)(best >> 32);
    const uint32_t mhi = __reduce_max_sync(mask, hi);
    const uint32_t mlo = __reduce_max_sync(mask, hi == mhi ? (uint32_t)best : 0u);
    if ((lane & 15) == 0 && b < a.B)
      group_best[b][0] = ((unsigned long long)mhi << 32) | mlo;
  }
}

}  // namespace
}  // namespace dspark
