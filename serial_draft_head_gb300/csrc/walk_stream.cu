// walk_stream.cu -- the persistent walk with NO residency: every step re-reads
// the CTA's W2 rows from L2/HBM.  It is the single-launch "L2 probe" of
// "Keeping the Draft Walk on Chip: One Launch for DSpark's Markov Head",
// section "V = 151,936: the whole bf16 table on chip" (the table read from L2
// every step inside one launch), and the path for any batch the resident
// kernel does not take.
//
// Layout: one CTA per SM, each owning a contiguous shard of vocabulary rows.
// A warp takes 32 consecutive rows, one row per lane: the lane streams its
// row (32 x 16 B) and dots it with u_b, read from shared memory as a
// broadcast, for NB requests at once.  No cross-lane reduction is needed, and
// the epilogue (two bf16 roundings, base add, score, key) runs per lane.
#include "walk_common.cuh"
#include "walk_kernels.h"

namespace dspark {

namespace {

constexpr int kStreamThreads = 512;
constexpr int kStreamWarps = kStreamThreads / 32;

__device__ __forceinline__ void unpack8(const uint4 w, float f[8]) {
  f[0] = __uint_as_float(w.x << 16);
  f[1] = __uint_as_float(w.x & 0xFFFF0000u);
  f[2] = __uint_as_float(w.y << 16);
  f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  f[4] = __uint_as_float(w.z << 16);
  f[5] = __uint_as_float(w.z & 0xFFFF0000u);
  f[6] = __uint_as_float(w.w << 16);
  f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
    x = y > x ? y : x;
  }
  return x;
}

// Projection + epilogue of this CTA's rows for requests [b0, b0 + NB).
template <int NB>
__device__ __forceinline__ void stream_rows(const WalkArgs& a, int k, int b0, int64_t row0,
                                            int64_t row1, const uint4* u_s, const float* temp_s,
                                            uint2 seed, unsigned long long* cta_key) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  unsigned long long best[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) best[j] = 0ull;

  for (int64_t rb = row0 + (int64_t)warp * 32; rb < row1; rb += (int64_t)kStreamWarps * 32) {
    const int64_t row = rb + lane;
    const bool valid = row < row1;
    const uint4* wrow = reinterpret_cast<const uint4*>(a.W2 + (valid ? row : row0) * kRank);
    float acc[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) acc[j] = 0.0f;
#pragma unroll 4
    for (int c = 0; c < kRank / 8; ++c) {
      float w[8];
      unpack8(__ldg(wrow + c), w);
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        float u[8];
        unpack8(u_s[(b0 + j) * (kRank / 8) + c], u);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j] = fmaf(w[e], u[e], acc[j]);
      }
    }
    if (valid) {
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int b = b0 + j;
        if (b < a.B) {
          const size_t off = ((size_t)b * a.gamma + k) * (size_t)a.V + (size_t)row;
          uint16_t lb;
          const unsigned long long key =
              epilogue_key(acc[j], a.base[off], temp_s[b], seed.x, seed.y, b, k,
                           (uint32_t)row, &lb);
          if (a.out_logits) a.out_logits[off] = lb;
          best[j] = key > best[j] ? key : best[j];
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const unsigned long long m = warp_max_u64(best[j]);
    if (lane == 0 && b0 + j < a.B && m != 0ull) atomicMax(&cta_key[b0 + j], m);
  }
}

template <int NB>
__global__ void __launch_bounds__(kStreamThreads, 1) walk_stream_kernel(const WalkArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int Bpad = (a.B + 7) & ~7;  // u rows past B are zero (read by the last group)
  uint4* u_s = reinterpret_cast<uint4*>(smem);                                     // [Bpad][32]
  unsigned long long* cta_key = reinterpret_cast<unsigned long long*>(smem + (size_t)Bpad * 512);
  int32_t* prev_s = reinterpret_cast<int32_t*>(cta_key + a.B);                     // [B]
  float* temp_s = reinterpret_cast<float*>(prev_s + a.B);                          // [B]
  __shared__ int flag_s;
  __shared__ uint32_t round_s;

  const int bad = check_inputs(a, &flag_s);
  if (bad != 0) {
    if (blockIdx.x == 0) {
      if (threadIdx.x == 0) set_status(a.sync.hdr, bad);
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    }
    return;
  }
  if (threadIdx.x == 0) round_s = *reinterpret_cast<volatile uint32_t*>(&a.sync.hdr->round);
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    prev_s[b] = a.anchor[b];
    temp_s[b] = a.temperature[b];
  }
  __syncthreads();
  const uint32_t parity = round_s & 1u;
  const uint2 eseed = round_seed(a, round_s);             // this round's Philox key
  if (blockIdx.x == 0) clear_other_parity(a.sync, parity);

  const int64_t row0 = (int64_t)blockIdx.x * a.rows_per_cta;
  const int64_t row1 = row0 + a.rows_per_cta < a.V ? row0 + a.rows_per_cta : a.V;

  bool ok = true;
  for (int k = 0; k < a.gamma && ok; ++k) {
    // u_b = W1[prev_b] for every request, into shared memory
    for (int i = threadIdx.x; i < Bpad * 32; i += blockDim.x) {
      const int b = i >> 5, c = i & 31;
      u_s[i] = b < a.B
                   ? __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)prev_s[b] * kRank) + c)
                   : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) cta_key[b] = 0ull;
    __syncthreads();
    for (int b0 = 0; b0 < a.B; b0 += NB)
      stream_rows<NB>(a, k, b0, row0, row1, u_s, temp_s, eseed, cta_key);
    __syncthreads();
    ok = exchange(a, round_s, k, cta_key, prev_s, &flag_s);
    if (ok && blockIdx.x == 0)
      for (int b = threadIdx.x; b < a.B; b += blockDim.x)
        a.out_tokens[(size_t)b * a.gamma + k] = prev_s[b];
  }
  if (blockIdx.x == 0) {
    if (!ok)
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    // every CTA read the round counter before its first post, and the last
    // rendezvous (or the error exit) is behind us: advance the parity
    if (threadIdx.x == 0) atomicAdd(&a.sync.hdr->round, 1u);
  }
}

}  // namespace

size_t stream_smem_bytes(int B) {
  const size_t Bpad = (size_t)((B + 7) & ~7);
  return Bpad * 512 + (size_t)B * 8 + (size_t)B * 4 + (size_t)B * 4;
}

int stream_threads() { return kStreamThreads; }

const void* stream_kernel_for(int B) {
  if (B >= 8) return reinterpret_cast<const void*>(&walk_stream_kernel<8>);
  if (B >= 4) return reinterpret_cast<const void*>(&walk_stream_kernel<4>);
  if (B >= 2) return reinterpret_cast<const void*>(&walk_stream_kernel<2>);
  return reinterpret_cast<const void*>(&walk_stream_kernel<1>);
}

namespace {

__global__ void gumbel_noise_kernel(const uint32_t* __restrict__ bits, float* __restrict__ noise,
                                    int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    noise[i] = gumbel_noise(bits[i]);
}

}  // namespace

cudaError_t gumbel_noise_launch(const uint32_t* bits, float* noise, int64_t n,
                                cudaStream_t stream) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  gumbel_noise_kernel<<<(unsigned)blocks, 256, 0, stream>>>(bits, noise, n);
  return cudaGetLastError();
}

}  // namespace dspark
