// walk_probe.cu -- dspark_walk_unit_rates: the per-SM rates at which the
// resident walk's three on-chip tiers feed the tensor cores, measured on the
// current device in SM clock cycles.  They are the unit costs of the walk's
// on-chip-read roofline: one step of the resident walk reads every row of the
// CTA's shard once ("Keeping the Draft Walk on Chip: One Launch for DSpark's
// Markov Head", section "B200: the bf16 table fits on chip": the table split
// over tensor memory, shared memory and registers, tcgen05 reading the
// tensor-memory part and mma.sync the rest).
//
// One CTA of 256 threads per SM (every SM busy, as in the walk) runs four
// timed phases, each between two CTA barriers:
//   1. mma.sync m16n8k16 with A in registers: 8 warps x 4 independent chains;
//   2. mma.sync with A read by ldmatrix from shared memory: 8 warps x 3 chains
//      over 16-row strips laid out as the walk's shared tier;
//   3. tcgen05.mma M=128 N=16 K=16 with A in tensor memory, issued by six
//      warps into their own accumulators (the walk's tensor-memory tier);
//   4. the projection of one walk step at the walk's shapes: the six warps
//      issue 8 tensor-memory MMAs each, then all warps run 16 k-tiles of 2
//      register and 3 shared-memory chains, then wait for the MMAs;
//   5. tcgen05.ld of mma.sync A fragments out of tensor memory: every warp
//      streams 256 columns of its lane quarter (32 KB) per pass;
//   6. the projection of one step when the tensor-memory tier feeds mma.sync
//      (4 strips per warp loaded by tcgen05.ld, 1 register strip, 3 shared
//      strips: 8 chains per warp over 16 k-tiles).
// Operand values are arbitrary (the rates do not depend on them); nothing of
// the walk is computed here.  Every wait is bounded by the global timer.
//
// A second kernel measures the two latencies that bound the walk's cross-SM
// rendezvous: how long after one SM's store another SM's poll sees it (CTA 0
// and one peer CTA bounce a counter through two words in separate lines;
// one-way time = round trip / 2, median over five peers), and the round trip
// of one dependent load that hits in L2.
#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/dspark_walk.h"
#include "tc_ptx.cuh"
#include "walk_common.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRfChains = 4;
constexpr int kRfIters = 2048;
constexpr int kSmChains = 3;
constexpr int kSmIters = 256;           // passes over the 16 k-tiles
constexpr int kIssuers = 6;
constexpr int kTcPerIssuer = 256;
constexpr int kStepReps = 64;
constexpr int kStrips = 8;              // shared strips of 16 rows x 256 K (8 KB)
constexpr int kStripBytes = 8192;
constexpr int kUBytes = 16 * 512;       // B operand: 16 columns x 256 K bf16
constexpr int kSmemBytes = 120 * 1024;  // one CTA per SM
constexpr int kPhases = 6;
constexpr int kLdReps = 64;
constexpr int64_t kWaitLimitNs = 100000000;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 16);

struct ProbeOut {
  long long cycles[kPhases];
  long long ns0;                 // global-timer ns of phase 1 (for the clock rate)
  int err;
  int pad;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint64_t t0) {
  uint32_t spins = 0;
  while (!ptx::mbar_try_wait(bar, parity))
    if ((++spins & 255u) == 0u && (int64_t)(globaltimer_ns() - t0) > kWaitLimitNs) return false;
  return true;
}

// Two bf16 values of magnitude in [1/8, 2) and random sign from a hash of i
// (operands like the walk's N(0, 1) weights; constant operands run faster).
__device__ __forceinline__ uint32_t rand_bf16x2(uint32_t i) {
  uint32_t h = i * 0x9E3779B1u;
  h ^= h >> 15;
  h *= 0x85EBCA77u;
  h ^= h >> 13;
  const uint32_t lo = 0x3E00u | ((h & 0x1u) << 15) | ((h >> 1) & 0x1FFu);
  const uint32_t hi = 0x3E00u | ((h & 0x400u) << 5) | ((h >> 11) & 0x1FFu);
  return lo | (hi << 16);
}

__global__ void __launch_bounds__(kThreads, 1) unit_rates_kernel(ProbeOut* out, float* sink,
                                                                 int random) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* strips = smem;                               // kStrips x 8 KB
  uint8_t* U = smem + kStrips * kStripBytes;            // 8 KB, 1024-aligned
  __shared__ __align__(8) uint64_t mbar[kIssuers];
  __shared__ uint32_t tmem_base_s;
  __shared__ int err_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < (kStrips * kStripBytes + kUBytes) / 4; i += kThreads)
    reinterpret_cast<uint32_t*>(smem)[i] = random ? rand_bf16x2((uint32_t)i) : 0x3F803F80u;
  if (threadIdx.x == 0) {
    err_s = 0;
    for (int i = 0; i < kIssuers; ++i) ptx::mbar_init(&mbar[i], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base_s, 512);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t u_addr = ptx::smem_u32(U);
  const uint32_t st_addr = ptx::smem_u32(strips);
  const uint32_t seed = threadIdx.x * 7u + blockIdx.x * 4099u;
  const uint32_t a0 = random ? rand_bf16x2(seed) : 0x3F803F80u ^ (uint32_t)lane;
  const uint32_t a1 = random ? rand_bf16x2(seed + 1u) : a0 + 1u;
  const uint32_t a2 = random ? rand_bf16x2(seed + 2u) : a0 + 2u;
  const uint32_t a3 = random ? rand_bf16x2(seed + 3u) : a0 + 3u;
  const uint32_t b0 = random ? rand_bf16x2(seed + 4u) : 0x3F803F80u;
  const uint32_t b1 = random ? rand_bf16x2(seed + 5u) : 0x3F803F80u;
  if (random) {       // tensor memory: every column of this warp's lane quarter
    uint32_t v[32];
    for (int c = 0; c < 256; c += 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = rand_bf16x2(seed * 613u + (uint32_t)(c + i));
      ptx::tmem_st32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256u * (uint32_t)(warp >> 2) + c, v);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
  }
  float sum = 0.0f;
  long long c0, c1;
  uint32_t commits = 0;      // completed phases of every issuer's mbarrier

  // 1. register-A mma.sync
  c0 = clock64();
  const uint64_t g0 = globaltimer_ns();
  {
    float acc[kRfChains][4] = {};
    for (int it = 0; it < kRfIters; ++it)
#pragma unroll
      for (int c = 0; c < kRfChains; ++c) ptx::mma_16816(acc[c], a0, a1, a2, a3, b0, b1);
#pragma unroll
    for (int c = 0; c < kRfChains; ++c) sum += acc[c][0] + acc[c][3];
  }
  __syncthreads();
  c1 = clock64();
  if (threadIdx.x == 0) {
    out[blockIdx.x].cycles[0] = c1 - c0;
    out[blockIdx.x].ns0 = (long long)(globaltimer_ns() - g0);
  }

  // 2. shared-memory-A mma.sync (ldmatrix of the walk's strip layout)
  const uint32_t blk0 = st_addr + (lane >> 3) * 128 + (lane & 7) * 16;
  __syncthreads();
  c0 = clock64();
  {
    float acc[kSmChains][4] = {};
    for (int it = 0; it < kSmIters; ++it)
#pragma unroll
      for (int kt = 0; kt < 16; ++kt)
#pragma unroll
        for (int j = 0; j < kSmChains; ++j) {
          uint32_t f0, f1, f2, f3;
          ptx::ldmatrix_x4(blk0 + (uint32_t)((warp + j) % kStrips) * kStripBytes + kt * 512, f0,
                           f1, f2, f3);
          ptx::mma_16816(acc[j], f0, f1, f2, f3, b0, b1);
        }
#pragma unroll
    for (int j = 0; j < kSmChains; ++j) sum += acc[j][0] + acc[j][3];
  }
  __syncthreads();
  c1 = clock64();
  if (threadIdx.x == 0) out[blockIdx.x].cycles[1] = c1 - c0;

  // 3. tensor-memory-A tcgen05.mma from six issuing warps
  __syncthreads();
  c0 = clock64();
  if (warp < kIssuers) {
    if (lane == 0) {
      const int t = warp >> 1;
      for (int i = 0; i < kTcPerIssuer; ++i) {
        const int kt = i & 15;
        const uint64_t bdesc = ptx::smem_desc_noswizzle(u_addr + kt * 512, 256, 128);
        ptx::tc_mma_tmem_a(tmem + 384 + 16 * warp, tmem + t * 128 + kt * 8, bdesc, kIdesc,
                           i > 0 ? 1u : 0u);
      }
      ptx::tc_commit(&mbar[warp]);
      if (!wait_bar(&mbar[warp], commits & 1u, globaltimer_ns())) err_s = 1;
    }
    __syncwarp();
  }
  ++commits;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  c1 = clock64();
  if (threadIdx.x == 0) out[blockIdx.x].cycles[2] = c1 - c0;

  // 4. one walk step's projection, repeated
  c0 = clock64();
  for (int rep = 0; rep < kStepReps && err_s == 0; ++rep) {
    if (warp < kIssuers && lane == 0) {
      const int t = warp >> 1, h = warp & 1;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int kt = 8 * h + kk;
        const uint64_t bdesc = ptx::smem_desc_noswizzle(u_addr + kt * 512, 256, 128);
        ptx::tc_mma_tmem_a(tmem + 384 + 16 * warp, tmem + t * 128 + kt * 8, bdesc, kIdesc,
                           kk > 0 ? 1u : 0u);
      }
      ptx::tc_commit(&mbar[warp]);
    }
    __syncwarp();
    float acc[2 + kSmChains][4] = {};
#pragma unroll
    for (int kt = 0; kt < 16; ++kt) {
      uint32_t af[kSmChains][4];
#pragma unroll
      for (int j = 0; j < kSmChains; ++j)
        ptx::ldmatrix_x4(blk0 + (uint32_t)((warp + j) % kStrips) * kStripBytes + kt * 512,
                         af[j][0], af[j][1], af[j][2], af[j][3]);
#pragma unroll
      for (int s = 0; s < 2; ++s) ptx::mma_16816(acc[s], a0 + kt, a1, a2, a3, b0, b1);
#pragma unroll
      for (int j = 0; j < kSmChains; ++j)
        ptx::mma_16816(acc[2 + j], af[j][0], af[j][1], af[j][2], af[j][3], b0, b1);
    }
#pragma unroll
    for (int s = 0; s < 2 + kSmChains; ++s) sum += acc[s][0];
    if (warp < kIssuers && lane == 0)
      if (!wait_bar(&mbar[warp], commits & 1u, globaltimer_ns())) err_s = 1;
    ++commits;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
  }
  c1 = clock64();
  if (threadIdx.x == 0) out[blockIdx.x].cycles[3] = (c1 - c0) / kStepReps;

  // 5. tensor memory -> registers: warp w reads lanes 32 (w % 4) .. + 31,
  // columns [256 (w / 4), + 256), 32 columns per load, two loads per wait
  const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tcol = 256u * (uint32_t)(warp >> 2);
  uint32_t xsum = 0u;
  __syncthreads();
  c0 = clock64();
  for (int rep = 0; rep < kLdReps; ++rep) {
#pragma unroll
    for (int c = 0; c < 8; c += 2) {
      uint32_t va[32], vb[32];
      ptx::tmem_ld32(tmem + tq + tcol + 32 * c, va);
      ptx::tmem_ld32(tmem + tq + tcol + 32 * c + 32, vb);
      ptx::tmem_wait_ld32(va);
      ptx::tmem_wait_ld32(vb);
#pragma unroll
      for (int i = 0; i < 32; ++i) xsum ^= va[i] + vb[i];
    }
  }
  __syncthreads();
  c1 = clock64();
  if (threadIdx.x == 0) out[blockIdx.x].cycles[4] = (c1 - c0) / kLdReps;

  // 6. one step's projection with the tensor-memory tier feeding mma.sync:
  // per k-tile pair one 32-column load (4 strips x 2 k-tiles x 4 words),
  // issued one pair ahead
  __syncthreads();
  c0 = clock64();
  for (int rep = 0; rep < kStepReps; ++rep) {
    float acc[8][4] = {};
    uint32_t fr[2][32];
    ptx::tmem_ld32(tmem + tq + tcol, fr[0]);
    ptx::tmem_wait_ld32(fr[0]);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p + 1 < 8) ptx::tmem_ld32(tmem + tq + tcol + 32 * (p + 1), fr[(p + 1) & 1]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int kt = 2 * p + h;
        uint32_t af[kSmChains][4];
#pragma unroll
        for (int j = 0; j < kSmChains; ++j)
          ptx::ldmatrix_x4(blk0 + (uint32_t)((warp + j) % kStrips) * kStripBytes + kt * 512,
                           af[j][0], af[j][1], af[j][2], af[j][3]);
        ptx::mma_16816(acc[0], a0 + kt, a1, a2, a3, b0, b1);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint32_t* f = &fr[p & 1][16 * h + 4 * s];
          ptx::mma_16816(acc[1 + s], f[0], f[1], f[2], f[3], b0, b1);
        }
#pragma unroll
        for (int j = 0; j < kSmChains; ++j)
          ptx::mma_16816(acc[5 + j], af[j][0], af[j][1], af[j][2], af[j][3], b0, b1);
      }
      if (p + 1 < 8) ptx::tmem_wait_ld32(fr[(p + 1) & 1]);
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) sum += acc[s][0];
  }
  __syncthreads();
  c1 = clock64();
  if (threadIdx.x == 0) {
    out[blockIdx.x].cycles[5] = (c1 - c0) / kStepReps;
    out[blockIdx.x].err = err_s;
  }
  if (xsum == 0x12345u) sink[blockIdx.x] = (float)xsum;
  if (sum == 1.2345f) sink[blockIdx.x] = sum;     // keeps the MMAs' results live
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

constexpr int kHopIters = 200;

__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// CTA 0 and CTA `peer` (one CTA per SM, co-resident: a cooperative launch)
// bounce a counter; CTA 0 then times a chain of dependent loads of a word
// that holds 0 (its own index).  words: [0] 0 -> peer, [32] peer -> 0, [64]
// the chained word.  out: [0] ns per one-way hop, [1] cycles per load.
__global__ void hop_kernel(uint32_t* words, int peer, long long* out, int* err) {
  if (threadIdx.x != 0) return;
  const int c = blockIdx.x;
  if (c != 0 && c != peer) return;
  uint32_t* a = words;
  uint32_t* b = words + 32;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i <= (uint32_t)kHopIters; ++i) {
    uint32_t spins = 0;
    if (c == 0) {
      st_relaxed_u32(a, i);
      while (ld_relaxed_gpu_u32(b) != i)
        if ((++spins & 1023u) == 0u && (int64_t)(globaltimer_ns() - t0) > kWaitLimitNs) {
          *err = 1;
          return;
        }
    } else {
      while (ld_relaxed_gpu_u32(a) != i)
        if ((++spins & 1023u) == 0u && (int64_t)(globaltimer_ns() - t0) > kWaitLimitNs) {
          *err = 1;
          return;
        }
      st_relaxed_u32(b, i);
    }
  }
  if (c != 0) return;
  out[0] = (long long)((globaltimer_ns() - t0) / (2ull * kHopIters));
  const uint32_t* w = words + 64;
  uint32_t idx = 0;
  const long long c0 = clock64();
  for (int i = 0; i < 1024; ++i) idx = ld_relaxed_gpu_u32(w + idx);
  out[1] = (clock64() - c0) / 1024 + (long long)(idx & 0x80000000u);
}

double median(std::vector<long long> v) {
  std::sort(v.begin(), v.end());
  const size_t n = v.size();
  return n % 2 ? (double)v[n / 2] : 0.5 * ((double)v[n / 2 - 1] + (double)v[n / 2]);
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" int dspark_walk_unit_rates(double* out, int n_out, void* stream) {
  if (!out || n_out < 5) return DSPARK_EINVAL;
  const int random = n_out >= 8 && out[7] != 0.0 ? 1 : 0;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSPARK_ECUDA;
  if (major != 10 || minor != 3) return DSPARK_EUNSUPPORTED;
  if (sms < 1 || sms > 1024) return DSPARK_EUNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProbeOut* d_out = nullptr;
  float* d_sink = nullptr;
  if (cudaMalloc(&d_out, sizeof(ProbeOut) * sms) != cudaSuccess) return DSPARK_ENOMEM;
  if (cudaMalloc(&d_sink, sizeof(float) * sms) != cudaSuccess) {
    cudaFree(d_out);
    return DSPARK_ENOMEM;
  }
  int rc = DSPARK_OK;
  std::vector<ProbeOut> h_out((size_t)sms);
  if (cudaFuncSetAttribute(unit_rates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess ||
      cudaMemsetAsync(d_out, 0, sizeof(ProbeOut) * sms, st) != cudaSuccess) {
    rc = DSPARK_ECUDA;
  } else {
    unit_rates_kernel<<<sms, kThreads, kSmemBytes, st>>>(d_out, d_sink, random);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(h_out.data(), d_out, sizeof(ProbeOut) * sms, cudaMemcpyDeviceToHost,
                        st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      rc = DSPARK_ECUDA;
  }
  cudaFree(d_out);
  cudaFree(d_sink);
  if (rc != DSPARK_OK) return rc;
  for (const ProbeOut& o : h_out)
    if (o.err) return DSPARK_ETIMEOUT;
  double med[kPhases + 1];
  std::vector<long long> v((size_t)sms);
  for (int p = 0; p < kPhases; ++p) {
    for (int i = 0; i < sms; ++i) v[i] = h_out[i].cycles[p];
    med[p] = median(v);
  }
  for (int i = 0; i < sms; ++i) v[i] = h_out[i].ns0;
  med[kPhases] = median(v);
  out[0] = med[0] / ((double)kWarps * kRfChains * kRfIters);
  out[1] = med[1] / ((double)kWarps * kSmChains * kSmIters * 16);
  out[2] = med[2] / ((double)kIssuers * kTcPerIssuer);
  out[3] = med[3];
  out[4] = med[kPhases] > 0 ? med[0] / med[kPhases] * 1000.0 : 0.0;   // cycles per us = MHz
  if (n_out >= 7) {
    out[5] = med[4] / 256.0;                 // 8 warps x 32 KB per rep: cycles per KB per SM
    out[6] = med[5];
  }
  if (n_out >= 10) {
    // cross-SM hop and L2 round trip: CTA 0 against five peers
    uint32_t* d_words = nullptr;
    long long* d_hop = nullptr;
    int* d_err = nullptr;
    if (cudaMalloc(&d_words, 512) != cudaSuccess) return DSPARK_ENOMEM;
    if (cudaMalloc(&d_hop, 2 * sizeof(long long)) != cudaSuccess ||
        cudaMalloc(&d_err, sizeof(int)) != cudaSuccess) {
      cudaFree(d_words);
      cudaFree(d_hop);
      return DSPARK_ENOMEM;
    }
    std::vector<long long> hop, rtt;
    const int peers[5] = {1, sms / 4, sms / 2, (3 * sms) / 4, sms - 1};
    if (cudaFuncSetAttribute(hop_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      rc = DSPARK_ECUDA;
    for (int pi = 0; pi < 5 && rc == DSPARK_OK && sms > 1; ++pi) {
      int peer = peers[pi] < 1 ? 1 : peers[pi];
      long long h[2] = {0, 0};
      int herr = 0;
      void* args[] = {&d_words, &peer, &d_hop, &d_err};
      if (cudaMemsetAsync(d_words, 0, 512, st) != cudaSuccess ||
          cudaMemsetAsync(d_err, 0, sizeof(int), st) != cudaSuccess ||
          cudaLaunchCooperativeKernel((const void*)hop_kernel, dim3(sms), dim3(32), args,
                                      kSmemBytes, st) != cudaSuccess ||
          cudaMemcpyAsync(h, d_hop, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
          cudaMemcpyAsync(&herr, d_err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess) {
        rc = DSPARK_ECUDA;
      } else if (herr) {
        rc = DSPARK_ETIMEOUT;
      } else {
        hop.push_back(h[0]);
        rtt.push_back(h[1]);
      }
    }
    cudaFree(d_words);
    cudaFree(d_hop);
    cudaFree(d_err);
    if (rc != DSPARK_OK) return rc;
    out[8] = hop.empty() ? 0.0 : median(hop);
    out[9] = rtt.empty() ? 0.0 : median(rtt);
  }
  return DSPARK_OK;
}
