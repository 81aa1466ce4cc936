// walk_kernels.h -- what the host side needs to know about each kernel.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {

// Streamed kernel (no residency): any batch up to kMaxB.
size_t stream_smem_bytes(int B);
int stream_threads();
const void* stream_kernel_for(int B);

// The kernels' Gumbel noise of n Philox words (a check of its arithmetic).
cudaError_t gumbel_noise_launch(const uint32_t* bits, float* noise, int64_t n,
                                cudaStream_t stream);

// Resident kernel: W2 tiered over tensor memory, registers, shared memory.
int64_t resident_words_per_cta(int RS, int S);
int resident_fixed_rows(int RS);
int resident_threads();
size_t resident_smem_bytes(int S, int ST, int nslot, int max_B, int R);
int resident_max_ring_slots();
const void* resident_kernel_for(int RS, int NT, bool cell);   // cell: recurrent heads / state output
int resident_max_smem_strips();
cudaError_t resident_repack(void* rowmajor, void* packed, int64_t V, int R, int RS, int S,
                            int n_cta, bool inverse, cudaStream_t stream);

// Resident kernel with every tier read by mma.sync (tensor memory through
// tcgen05.ld): batches up to mma_resident_max_batch(), the Markov head.
// Shards of at most mma_resident_max_rows() rows stay on chip; larger ones
// keep S shared strips per CTA and stream ST more every step through a ring
// of nslot half-strip slots per warp (S and ST multiples of 8).
int mma_resident_fixed_rows();
int mma_resident_max_rows();
int mma_resident_max_batch();
int mma_resident_max_ctas();                  // the grid's largest size
int64_t mma_resident_words_per_cta(int S);    // S: every strip in the shared-tier format
size_t mma_resident_smem_bytes(int S, int max_B, int R, int nslot);
// S shared strips, NT n-tiles (B <= 8 NT), a streamed tier or not
const void* mma_resident_kernel(int S, int NT, bool streamed);
cudaError_t mma_resident_repack(void* rowmajor, void* packed, int64_t V, int R, int S, int n_cta,
                                bool inverse, cudaStream_t stream);

// Batched kernel: W2 streamed through a TMA ring, tcgen05 with N = B.
struct WalkArgs;
int batched_threads();
size_t batched_smem_bytes(int nst, int N);
int batched_max_stages();
const void* batched_kernel();
cudaError_t batched_repack(void* rowmajor, void* packed, int64_t V, int R, int n_cta,
                           bool inverse, cudaStream_t stream);
cudaError_t batched_launch(const WalkArgs& w, const void* W2b, int R, int n_cta, int max_B, int B,
                           size_t smem_budget, cudaStream_t stream);

}  // namespace dspark
