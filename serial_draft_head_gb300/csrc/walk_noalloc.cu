// walk_noalloc.cu -- dspark_walk_run_noalloc: one round of the streamed walk
// for callers that must not allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside an
// allocator's own callbacks, in a process whose device memory is entirely
// owned by a caching pool that other code must not bypass, or on a path that
// must never block on the driver's allocator (whose calls can synchronise
// the device).  Such callers cannot create a handle (dspark_walk_create
// allocates the repacked weights and the rendezvous slots), so this entry
// point reads W2 from the caller's own buffer and keeps the rendezvous slots
// in a fixed block of device memory that the library image carries.
//
// The block is a file-scope __device__ array, so every GPU that loads this
// library holds it (kScratchBytes below, about 17.5 KB) until the process exits.
// A __device__ variable's address belongs to a CUDA context, and host code
// cannot use the array's name as a device address.  So every call looks the
// address up in the caller's current context with cudaGetSymbolAddress (a
// lookup, no allocation), and makes sure the streamed kernels it may launch
// are loaded (cudaFuncGetAttributes): the entry point follows the caller's
// context, including a context created anew after cudaDeviceReset.  The first
// call in a context is where the driver loads these kernels (with lazy module
// loading, the default, that can allocate and synchronise), so make it once
// before capturing any stream into a CUDA graph or entering code that must
// not allocate.
//
// All calls share the one block: each call clears it on its stream before
// launching, so calls that overlap on the GPU (different streams without an
// ordering between them) race on it and must not be issued.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dspark_walk.h"
#include "walk_common.cuh"
#include "walk_kernels.h"

using namespace dspark;

namespace {

constexpr int kNoAllocMaxB = 64;
constexpr int kNoAllocMaxGamma = 16;
constexpr size_t kCountOff = 128;  // after the 32-byte header, 128-byte aligned
constexpr size_t kKeyOff =
    kCountOff + (size_t)2 * kNoAllocMaxGamma * kCountStride * sizeof(uint32_t);
constexpr size_t kScratchBytes =
    kKeyOff + (size_t)2 * kNoAllocMaxGamma * kNoAllocMaxB * sizeof(unsigned long long);
static_assert(kKeyOff % 128 == 0, "key slots must stay aligned");

// The rendezvous state of dspark_walk_run_noalloc (header, arrival counts,
// 64-bit keys), one copy per device that loads the library.
static __device__ __align__(256) unsigned char g_walk_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceCheck {
  std::once_flag once;
  int rc = DSPARK_OK;
  int sm_count = 0;
};

DeviceCheck g_check[kMaxDevices];

// Once per device: the device is an sm_103 part that can run cooperative
// kernels (properties of the device, not of a context).
void check_device(DeviceCheck* s, int dev) {
  int major = 0, minor = 0, sms = 0, coop = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
    s->rc = DSPARK_ECUDA;
    return;
  }
  if (major != 10 || minor != 3 || !coop) {
    s->rc = DSPARK_EUNSUPPORTED;
    return;
  }
  s->sm_count = sms;
  s->rc = DSPARK_OK;
}

// In the current context: the scratch block's device address, and the four
// streamed-kernel instantiations loaded.  Allocates nothing itself.
int resolve_in_context(void** scratch) {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_walk_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    return DSPARK_ECUDA;
  }
  for (int b = 1; b <= 8; b *= 2) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, stream_kernel_for(b)) != cudaSuccess) {
      cudaGetLastError();
      return DSPARK_ECUDA;
    }
  }
  *scratch = ptr;
  return DSPARK_OK;
}

}  // namespace

extern "C" int dspark_walk_run_noalloc(const void* W1, const void* W2, int64_t V, int r,
                                       const void* base_logits, const int32_t* anchor,
                                       const float* temperature, uint64_t seed,
                                       int32_t* out_tokens, int B, int gamma, void* out_logits,
                                       void* stream) {
  if (!W1 || !W2 || !base_logits || !anchor || !temperature || !out_tokens) return DSPARK_EINVAL;
  if (r != kRank) return DSPARK_EUNSUPPORTED;
  if (V < 1 || V >= ((int64_t)1 << 31) || B < 1 || gamma < 1) return DSPARK_EINVAL;
  if (B > kNoAllocMaxB || gamma > kNoAllocMaxGamma) return DSPARK_ELIMIT;
  if ((reinterpret_cast<uintptr_t>(W1) & 15u) != 0 || (reinterpret_cast<uintptr_t>(W2) & 15u) != 0)
    return DSPARK_EINVAL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSPARK_EUNSUPPORTED;
  DeviceCheck* s = &g_check[dev];
  std::call_once(s->once, check_device, s, dev);
  if (s->rc != DSPARK_OK) return s->rc;
  void* scratch = nullptr;
  const int rc = resolve_in_context(&scratch);
  if (rc != DSPARK_OK) return rc;

  // shard plan: at least 32 rows per CTA, at most one CTA per SM
  int64_t n = (V + 31) / 32;
  if (n > s->sm_count) n = s->sm_count;
  if (n < 1) n = 1;
  const int64_t rpc = (V + n - 1) / n;
  n = (V + rpc - 1) / rpc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the previous call's state is still in the block: start from zero
  if (cudaMemsetAsync(scratch, 0, kScratchBytes, st) != cudaSuccess) return DSPARK_ECUDA;

  uint8_t* base = static_cast<uint8_t*>(scratch);
  WalkArgs a{};
  a.W1 = static_cast<const uint16_t*>(W1);
  a.W2 = static_cast<const uint16_t*>(W2);
  a.base = static_cast<const uint16_t*>(base_logits);
  a.anchor = anchor;
  a.temperature = temperature;
  a.out_tokens = out_tokens;
  a.out_logits = static_cast<uint16_t*>(out_logits);
  a.sync.hdr = reinterpret_cast<SyncHeader*>(base);
  a.sync.count = reinterpret_cast<uint32_t*>(base + kCountOff);
  a.sync.key = reinterpret_cast<unsigned long long*>(base + kKeyOff);
  a.sync.max_gamma = kNoAllocMaxGamma;
  a.sync.max_B = kNoAllocMaxB;
  a.V = V;
  a.B = B;
  a.gamma = gamma;
  a.rows_per_cta = (int)rpc;
  a.seed_lo = (uint32_t)seed;
  a.seed_hi = (uint32_t)(seed >> 32);
  a.timeout_ns = 200000000;
  a.skip_cta = -1;

  // at most 64 requests: the kernel's shared memory stays under the 48 KB
  // that needs no opt-in attribute
  const void* fn = stream_kernel_for(B);
  void* args[] = {&a};
  if (cudaLaunchCooperativeKernel(fn, dim3((unsigned)n), dim3(stream_threads()), args,
                                  stream_smem_bytes(B), st) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}
