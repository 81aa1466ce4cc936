// walk_kernels.h -- what the host side needs to know about each kernel.
#pragma once
#include <stddef.h>

namespace dspark {

// Streamed kernel (no residency): any batch up to kMaxB.
size_t stream_smem_bytes(int B);
int stream_threads();
const void* stream_kernel_for(int B);

}  // namespace dspark
