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
// CTA = 8 epilogue warps + 1 control warp.  The control warp's lane 0 keeps
// NST half-tiles (32 KB: 128 rows x 128 K) of the CTA's W2 shard in flight
// with cp.async.bulk, issues the 8 MMAs of each half-tile into one of two
// TMEM accumulators (128 x N fp32 each), and commits them to mbarriers.  The
// epilogue warps read a finished accumulator (warp w: lane quarter w % 4,
// column half w / 4), apply the fused epilogue (two bf16 roundings, base add,
// score), fold keys per request, and free the accumulator.  After the last
// tile the CTA's best key per request goes through the atomic rendezvous and
// the next u rows are gathered into U.
#include "tc_ptx.cuh"
#include "walk_common.cuh"
#include "walk_kernels.h"

namespace dspark {

namespace {

constexpr int kEpiWarps = 8;
constexpr int kBatThreads = (kEpiWarps + 1) * 32;
constexpr int kStageBytes = 32768;            // half a tile: 128 rows x 128 K bf16
constexpr int kBlockBytes = 4096;             // 128 rows x 16 K
constexpr int kMaxStages = 6;

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

// Maximum of a 64-bit key over the lanes of `mask` with two redux.sync.
__device__ __forceinline__ unsigned long long group_max_key(unsigned mask, unsigned long long key) {
  const uint32_t hi = (uint32_t)(key >> 32);
  const uint32_t mhi = __reduce_max_sync(mask, hi);
  const uint32_t mlo = __reduce_max_sync(mask, hi == mhi ? (uint32_t)key : 0u);
  return ((unsigned long long)mhi << 32) | mlo;
}

// u_b = W1[tok] into U (core matrix (kc, b / 8) at (kc * N/8 + b/8) * 128).
// Eight rows' chunks in flight per thread before any store.
__device__ __forceinline__ void gather_u(const WalkArgs& a, const int32_t* tok_s, uint8_t* U,
                                         int N) {
  const int epi_threads = kEpiWarps * 32;
  const int total = a.B * 32;
  for (int i0 = threadIdx.x; i0 < total; i0 += 8 * epi_threads) {
    uint4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * epi_threads;
      if (i < total)
        x[u] = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok_s[i >> 5] * kRank) +
                     (i & 31));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * epi_threads;
      if (i < total) {
        const int b = i >> 5, c = i & 31;
        *reinterpret_cast<uint4*>(U + ((size_t)c * (N >> 3) + (b >> 3)) * 128 + (b & 7) * 16) =
            x[u];
      }
    }
  }
  ptx::fence_proxy_async_smem();
}

__global__ void __launch_bounds__(kBatThreads, 1) walk_batched_kernel(const BatchedArgs ba) {
  const WalkArgs& a = ba.w;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int N = ba.N;
  uint8_t* ring = smem;                                            // nst x 32 KB
  uint8_t* U = smem + (size_t)ba.nst * kStageBytes;                // N x 512 B
  unsigned long long* wbest = reinterpret_cast<unsigned long long*>(U + (size_t)N * 512);
  // wbest: [8 warps][128] running best per (warp, request in the warp's half)
  unsigned long long* cta_key = wbest + kEpiWarps * 128;           // [256]
  int32_t* tok_s = reinterpret_cast<int32_t*>(cta_key + 256);      // [256]
  float* temp_s = reinterpret_cast<float*>(tok_s + 256);           // [256]
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
  if (warp < kEpiWarps) gather_u(a, tok_s, U, N);

  // control state (lane 0 of the control warp)
  const int stages_total = 2 * T * a.gamma;   // half-tiles consumed this round
  int issued = 0;                             // half-tiles whose copy was issued
  if (warp == kEpiWarps && lane == 0) {
    const int pre = nst < stages_total ? nst : stages_total;
    for (; issued < pre; ++issued) {
      const int gl = issued % (2 * T);
      ptx::mbar_expect_tx(&full_bar[issued % nst], kStageBytes);
      ptx::bulk_g2s(ring + (size_t)(issued % nst) * kStageBytes, gw + (size_t)gl * kStageBytes,
                    kStageBytes, &full_bar[issued % nst]);
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
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
              const int kt = 8 * h + j;
              const uint64_t adesc = ptx::smem_desc_noswizzle(
                  ring_addr + (uint32_t)s * kStageBytes + (uint32_t)j * kBlockBytes, 2048, 128);
              const uint64_t bdesc =
                  ptx::smem_desc_noswizzle(u_addr + (uint32_t)kt * 32u * (uint32_t)N,
                                           16u * (uint32_t)N, 128);
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
                      tmem + (uint32_t)(d * 256)),
                  "l"(adesc), "l"(bdesc), "r"(idesc), "r"(kt > 0 ? 1u : 0u)
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
              ptx::bulk_g2s(ring + (size_t)ps * kStageBytes, gw + (size_t)gl * kStageBytes,
                            kStageBytes, &full_bar[ps]);
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
      // warp w: rows 32 (w % 4) .. +31 of every tile, columns (requests)
      // [c0, c0 + cols).  Base logits come from HBM: the loads of the next
      // 16-column chunk are issued before the current chunk is computed.
      const int q = warp & 3, half = warp >> 2;
      const int cols = N >> 1;
      const int c0 = half * cols;
      int act = a.B - c0;                            // this warp's live columns
      act = act < 0 ? 0 : (act > cols ? cols : act);
      const int cpt = (act + 15) >> 4;               // chunks per tile
      const int nc = cpt * T;
      for (int i = lane; i < 128; i += 32) wbest[warp * 128 + i] = 0ull;
      __syncwarp();
      uint32_t nxt[16];
      auto prefetch = [&](int ci) {
        const int t = ci / cpt, cb = (ci - t * cpt) * 16;
        const int64_t v = row0 + t * 128 + 32 * q + lane;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int b = c0 + cb + j;
          nxt[j] = (cb + j < act && v < a.V)
                       ? (uint32_t)__ldg(a.base + ((size_t)b * a.gamma + k) * (size_t)a.V + v)
                       : 0u;
        }
      };
      if (nc > 0) prefetch(0);
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
        const int64_t v = row0 + t * 128 + 32 * q + lane;
        const bool valid = v < a.V;
        for (int cc = 0; cc < cpt; ++cc, ++ci) {
          const int cb = cc * 16;
          uint32_t cur[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) cur[j] = nxt[j];
          if (ci + 1 < nc) prefetch(ci + 1);
          uint32_t dv[16];
          ptx::tmem_ld<16>(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * 256 + c0 + cb), dv);
          ptx::tmem_wait_ld();
          // 8 keys at a time first (independent chains the compiler can
          // interleave), then their warp reductions
#pragma unroll
          for (int j0 = 0; j0 < 16; j0 += 8) {
            unsigned long long key[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj;
              const int b = c0 + cb + j;
              key[jj] = 0ull;
              if (cb + j < act && valid) {
                const float bias = __bfloat162float(__float2bfloat16_rn(__uint_as_float(dv[j])));
                const uint16_t lb =
                    float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(cur[j]), bias));
                if (a.out_logits)
                  a.out_logits[((size_t)b * a.gamma + k) * (size_t)a.V + (size_t)v] = lb;
                const float T_b = temp_s[b];
                const float logit = bf16_bits_to_float(lb);
                float sc = logit;
                if (T_b > 0.0f) {
                  const uint4 r = philox4x32_10(make_uint4((uint32_t)v >> 2, (uint32_t)k,
                                                           (uint32_t)b, 0u),
                                                a.seed_lo, a.seed_hi);
                  sc = gumbel_score(logit, T_b, philox_word(r, (uint32_t)v & 3u));
                }
                key[jj] = make_key(sc, (uint32_t)v);
              }
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = j0 + jj;
              if (cb + j >= act) continue;           // uniform across the warp
              const unsigned long long m = group_max_key(0xFFFFFFFFu, key[jj]);
              if (lane == 0) {
                unsigned long long* p = &wbest[warp * 128 + (cb + j)];
                *p = m > *p ? m : *p;
              }
            }
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

    // CTA best per request: max over the 4 lane quarters of its column half
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
      const int half = b / (N >> 1), j = b - half * (N >> 1);
      unsigned long long m = 0ull;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const unsigned long long x = wbest[(half * 4 + qq) * 128 + j];
        m = x > m ? x : m;
      }
      cta_key[b] = m;
    }
    __syncthreads();
    trace_stamp(a, k, 4);
    ok = exchange(a, round_s, k, cta_key, tok_s, &flag_s);
    trace_stamp(a, k, 5);
    if (!ok) break;
    if (cta == 0)
      for (int b = threadIdx.x; b < a.B; b += blockDim.x)
        a.out_tokens[(size_t)b * a.gamma + k] = tok_s[b];
    if (k + 1 < a.gamma && warp < kEpiWarps) gather_u(a, tok_s, U, N);
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
__global__ void repack_batched_kernel(const uint32_t* __restrict__ W2w, uint32_t* __restrict__ out,
                                      int64_t V, int R, int64_t total_words) {
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
    out[i] = row < V ? W2w[row * (kRank / 2) + kp] : 0u;
  }
}

}  // namespace

int batched_threads() { return kBatThreads; }

size_t batched_smem_bytes(int nst, int N) {
  return (size_t)nst * kStageBytes + (size_t)N * 512 + (size_t)kEpiWarps * 128 * 8 + 256 * 8 +
         256 * 4 + 256 * 4;
}

int batched_max_stages() { return kMaxStages; }

const void* batched_kernel() { return reinterpret_cast<const void*>(&walk_batched_kernel); }

cudaError_t batched_repack(const void* W2, void* out, int64_t V, int R, int n_cta,
                           cudaStream_t stream) {
  const int64_t total = (int64_t)n_cta * (R / 128) * 16 * 1024;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  repack_batched_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint32_t*>(W2),
                                                    static_cast<uint32_t*>(out), V, R, total);
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
