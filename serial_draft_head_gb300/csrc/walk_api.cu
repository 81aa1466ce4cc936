// walk_api.cu -- the C ABI of include/dspark_walk.h: argument checks, the
// shard plan, device allocations owned by a handle, and the cooperative
// launch of one persistent kernel per round.
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "../../include/dspark_walk.h"
#include "walk_common.cuh"
#include "walk_kernels.h"

using namespace dspark;

struct dspark_walk {
  int device = 0;
  int sm_count = 0;
  int64_t V = 0;
  int r = 0;
  int max_B = 0;
  int max_gamma = 0;
  const uint16_t* W1 = nullptr;   // caller-owned
  // W2 is kept only in the layouts the runs need, each built when first
  // needed (the row-major copy only for the streamed kernel); any missing
  // layout is rebuilt from one that exists.
  uint16_t* W2 = nullptr;         // row-major copy (streamed kernel)
  void* sync_mem = nullptr;       // SyncHeader + counts + keys + resident slots
  SyncView sync{};
  // mma.sync resident layout (Markov runs with B <= mr_max_B)
  uint32_t* W2m = nullptr;
  bool mr_ok = false;             // the layout can hold the shard
  int mr_max_B = 0, mr_R = 0, mr_S = 0, mr_n_cta = 0;
  int mr_ST = 0, mr_nslot = 0;    // streamed strips per CTA, ring slots per warp
  int64_t mr_wpc = 0;
  size_t mr_smem = 0;
  // tcgen05 resident layout (runs with B <= res_max_B the layout above does
  // not take: the recurrent heads and the state output)
  uint32_t* W2p = nullptr;        // tiered repack, res_wpc words per CTA
  int res_max_B = 0;              // 0: no resident placement
  bool use_resident = true;       // dspark_walk_set_kernel
  int seed_per_round = 0;         // dspark_walk_set_seed_mode
  int sampler = 0;                // dspark_walk_set_sampler
  int cell = 0;                   // dspark_walk_set_cell
  const uint16_t* cell_M = nullptr;   // caller-owned [256, 256] ([768, 256] for the GRU)
  const uint16_t* cell_X = nullptr;   // caller-owned GRU token tables [3, V, 256]
  float* cell_p = nullptr;        // handle-owned [max_gamma][16][kCellP] fp32
  uint16_t* out_state = nullptr;  // caller-owned, dspark_walk_set_state_output
  int res_RS = 0, res_NT = 0, res_R = 0, res_S = 0, res_ST = 0, res_nslot = 0, res_n_cta = 0;
  int64_t res_wpc = 0;
  size_t res_smem = 0;
  dspark_walk_plan plan{};
  int st_n_cta = 0, st_rpc = 0;   // streamed kernel's shard plan
  // batched layout (runs the resident kernel does not take)
  uint8_t* W2b = nullptr;
  int bat_R = 0, bat_n_cta = 0;
  bool use_batched = true;
  int64_t timeout_ns = 200000000;
  unsigned long long* trace = nullptr;  // caller-owned, see dspark_walk_set_trace
  int64_t trace_bytes = 0;
  int trace_global = 0;                 // dspark_walk_set_trace_clock
  int skip_cta = -1;
  // staging for dspark_walk_run_host (allocated on first use): device, and a
  // pinned host block {anchor[max_B], temperature[max_B], status}
  void* stage = nullptr;
  size_t stage_bytes = 0;
  void* hstage = nullptr;
};

namespace {

int cuda_fail(cudaError_t e) {
  if (e == cudaErrorMemoryAllocation) return DSPARK_ENOMEM;
  return DSPARK_ECUDA;
}

#define CUDA_TRY(expr)                                 \
  do {                                                 \
    cudaError_t err_ = (expr);                         \
    if (err_ != cudaSuccess) return cuda_fail(err_);   \
  } while (0)

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sizes of the parts of the rendezvous memory: header, arrival counts, keys,
// tagged slots (slot_B requests, slot_stride words per step and request).
void sync_layout(int max_gamma, int max_B, int slot_B, int slot_stride, size_t* count_off,
                 size_t* key_off, size_t* slot_off, size_t* total) {
  *count_off = round_up(sizeof(SyncHeader), 128);
  *key_off = round_up(*count_off + (size_t)2 * max_gamma * kCountStride * sizeof(uint32_t), 128);
  *slot_off = round_up(*key_off + (size_t)2 * max_gamma * max_B * sizeof(unsigned long long), 128);
  *total = round_up(*slot_off + (size_t)2 * max_gamma * slot_B * slot_stride *
                                    sizeof(unsigned long long), 128);
}

// Shared memory a CTA may use, minus the kernels' static shared variables.
constexpr size_t kSmemBudget = 232448 - 2048;

// Batched plan: rows spread over at most one CTA per SM in whole 128-row
// tiles; every step streams the CTA's tiles through the TMA ring.
void plan_batched(dspark_walk* h) {
  int64_t R = (h->V + h->sm_count - 1) / h->sm_count;
  R = (R + 127) / 128 * 128;
  h->bat_R = (int)R;
  h->bat_n_cta = (int)((h->V + R - 1) / R);
}

// Resident plan: every CTA holds 3 tensor-memory tiles (384 rows), 2
// register strips per warp (256 rows) and S <= 24 shared-memory strips; rows
// are spread evenly over at most one CTA per SM (R a multiple of 16).  When
// the shard does not fit, the rows left over are streamed: ST strips per CTA
// go through a two-slot ring of 64 KB bulk copies every step (the slots that
// ring needs come out of the shared-memory tier), as in "V = 248,320: 62% on
// chip, the rest streamed".  Returns false when B or V are too large, in which
// case every run uses the batched or streamed kernel.
bool plan_resident(dspark_walk* h) {
  const int mb = h->max_B < 16 ? h->max_B : 16;
  if (h->V >= (1 << 18)) return false;          // the 18-bit id field of the slot word
  const int RS = 2;
  const int NT = mb <= 8 ? 1 : 2;
  const int fixed = resident_fixed_rows(RS);
  int64_t R = (h->V + h->sm_count - 1) / h->sm_count;
  R = (R + 15) / 16 * 16;
  if (R < fixed) R = fixed;
  const int S_all = (int)((R - fixed) / 16);
  int S = S_all, ST = 0, nslot = 0;
  if (S > resident_max_smem_strips() || resident_smem_bytes(S, 0, 0, mb, (int)R) > kSmemBudget) {
    // as many ring slots as fit (more bytes in flight), then shared strips
    for (nslot = resident_max_ring_slots(); nslot >= 2; --nslot)
      if (resident_smem_bytes(0, 1, nslot, mb, (int)R) <= kSmemBudget) break;
    if (nslot < 2) return false;
    const size_t other = resident_smem_bytes(0, 1, nslot, mb, (int)R);
    S = (int)((kSmemBudget - other) / 8192);
    if (S > resident_max_smem_strips()) S = resident_max_smem_strips();
    if (S > S_all) S = S_all;
    ST = S_all - S;
  }
  h->res_max_B = mb;
  h->res_RS = RS;
  h->res_NT = NT;
  h->res_R = (int)R;
  h->res_S = S;
  h->res_ST = ST;
  h->res_nslot = nslot;
  h->res_n_cta = (int)((h->V + R - 1) / R);
  h->res_wpc = resident_words_per_cta(RS, S + ST);
  h->res_smem = resident_smem_bytes(S, ST, nslot, mb, (int)R);
  return true;
}

// mma.sync resident plan: rows spread over at most one CTA per SM, each CTA
// holding 512 rows in tensor memory, 128 in registers and 0, 128, 256 or 384
// in shared memory (the same number of shared strips in every warp), so shards
// of 640 .. 1,024 rows: V <= 155,648 on 152 SMs.  Larger shards keep tensor
// memory, registers and NS = 0..2 shared strips per warp, and stream the rest
// (ST strips per CTA, one of every warp per item) every step through a ring of
// nslot = 2 or 3 slots of 64 KB, as in "V = 248,320: 62% on chip, the rest
// streamed": the most shared strips that fit first, then the most slots.
bool plan_mma(dspark_walk* h) {
  if (h->V >= (1 << 18)) return false;          // the 18-bit id field of the slot word
  const int mb = h->max_B < mma_resident_max_batch() ? h->max_B : mma_resident_max_batch();
  const int fixed = mma_resident_fixed_rows();
  int64_t R0 = (h->V + h->sm_count - 1) / h->sm_count;
  R0 = (R0 + 15) / 16 * 16;
  if (R0 < fixed) R0 = fixed;
  int64_t R = 0;
  int S = 0, ST = 0, nslot = 0;
  if (R0 <= mma_resident_max_rows()) {
    // every warp runs the same number NS of shared strips: R = 640 + 128 NS, or
    // one strip less when the batch's base rows would not fit otherwise (the
    // last warp's third strip then only pads, over the U buffer that follows)
    R = fixed + (R0 - fixed + 127) / 128 * 128;
    if (mma_resident_smem_bytes((int)((R - fixed) / 16), mb, (int)R, 0) > kSmemBudget &&
        R > fixed && R - 16 >= R0)
      R -= 16;
    S = (int)((R - fixed) / 16);
  } else {
    for (int ns = 2; ns >= 0 && nslot == 0; --ns)
      for (int sl = 3; sl >= 2; --sl) {
        const int64_t kept = fixed + 128 * ns;
        R = kept + (R0 - kept + 127) / 128 * 128;
        if (R >= 65536) return false;           // the 16-bit local row of the CTA's keys
        if (mma_resident_smem_bytes(8 * ns, mb, (int)R, sl) <= kSmemBudget) {
          S = 8 * ns;
          ST = (int)((R - kept) / 16);
          nslot = sl;
          break;
        }
      }
    if (nslot == 0) return false;
  }
  const size_t smem = mma_resident_smem_bytes(S, mb, (int)R, nslot);
  if (smem > kSmemBudget) return false;
  if ((h->V + R - 1) / R > mma_resident_max_ctas()) return false;
  h->mr_ok = true;
  h->mr_max_B = mb;
  h->mr_R = (int)R;
  h->mr_S = S;
  h->mr_ST = ST;
  h->mr_nslot = nslot;
  h->mr_n_cta = (int)((h->V + R - 1) / R);
  h->mr_wpc = mma_resident_words_per_cta(S + ST);
  h->mr_smem = smem;
  return true;
}

// Shard plan of the streamed kernel: rows split evenly over at most one CTA
// per SM; tiny vocabularies use fewer CTAs (at least 32 rows each), since
// the rendezvous costs more with more CTAs.
void plan_stream(dspark_walk* h) {
  const int64_t min_rows = 32;
  int64_t n = (h->V + min_rows - 1) / min_rows;
  if (n > h->sm_count) n = h->sm_count;
  if (n < 1) n = 1;
  int64_t rpc = (h->V + n - 1) / n;
  n = (h->V + rpc - 1) / rpc;     // every CTA owns at least one row
  h->st_n_cta = (int)n;
  h->st_rpc = (int)rpc;
  dspark_walk_plan& p = h->plan;
  p.V = h->V;
  p.r = h->r;
  p.n_cta = (int)n;
  p.threads = stream_threads();
  p.rows_per_cta = (int)rpc;
  p.rows_tmem = p.rows_smem = p.rows_rf = 0;
  p.rows_stream = (int)rpc;
  p.resident_bytes = 0;
  p.streamed_bytes = h->V * (int64_t)h->r * 2;
  p.max_B = h->max_B;
  p.max_gamma = h->max_gamma;
  p.kernel = DSPARK_KERNEL_STREAM;
  p.sm_count = h->sm_count;
  if (h->mr_ok) {
    p.n_cta = h->mr_n_cta;
    p.threads = resident_threads();
    p.rows_per_cta = h->mr_R;
    p.rows_tmem = 512;
    p.rows_rf = 128;
    p.rows_smem = 16 * h->mr_S;
    p.rows_stream = 16 * h->mr_ST;
    p.streamed_bytes = (int64_t)16 * h->mr_ST * h->mr_n_cta * h->r * 2;
    p.resident_bytes = h->V * (int64_t)h->r * 2 - p.streamed_bytes;
    if (p.resident_bytes < 0) p.resident_bytes = 0;
    p.kernel = DSPARK_KERNEL_RESIDENT;
  } else if (h->res_max_B > 0) {
    p.n_cta = h->res_n_cta;
    p.threads = resident_threads();
    p.rows_per_cta = h->res_R;
    p.rows_tmem = 384;
    p.rows_rf = 128 * h->res_RS;
    p.rows_smem = 16 * h->res_S;
    p.rows_stream = 16 * h->res_ST;
    p.streamed_bytes = (int64_t)16 * h->res_ST * h->res_n_cta * h->r * 2;
    p.resident_bytes = h->V * (int64_t)h->r * 2 - p.streamed_bytes;
    if (p.resident_bytes < 0) p.resident_bytes = 0;
    p.kernel = DSPARK_KERNEL_RESIDENT;
  }
}

// ------------------------------------------------------- W2 layouts ----
// Which layout a Markov run of B requests takes, given the kernel choice.
enum class Path { kMma, kResident, kBatched, kStream };

bool cell_run(const dspark_walk* h) {
  return h->cell != DSPARK_CELL_MARKOV || h->out_state != nullptr;
}

Path path_for(const dspark_walk* h, int B) {
  if (h->use_resident) {
    if (h->mr_ok && !cell_run(h) && B <= h->mr_max_B) return Path::kMma;
    if (h->res_max_B > 0 && B <= h->res_max_B) return Path::kResident;
  }
  if (h->use_batched) return Path::kBatched;
  return Path::kStream;
}

size_t rowmajor_bytes(const dspark_walk* h) { return (size_t)h->V * h->r * 2; }

// Row-major W2 into `dst` from any layout the handle holds.
cudaError_t unpack_rowmajor(dspark_walk* h, void* dst) {
  if (h->W2) return cudaMemcpy(dst, h->W2, rowmajor_bytes(h), cudaMemcpyDeviceToDevice);
  if (h->W2m)
    return mma_resident_repack(dst, h->W2m, h->V, h->mr_R, h->mr_S + h->mr_ST, h->mr_n_cta, true,
                               0);
  if (h->W2p)
    return resident_repack(dst, h->W2p, h->V, h->res_R, h->res_RS, h->res_S + h->res_ST,
                           h->res_n_cta, true, 0);
  if (h->W2b) return batched_repack(dst, h->W2b, h->V, h->bat_R, h->bat_n_cta, true, 0);
  return cudaErrorInvalidValue;
}

// Build the layout `which` from row-major W2 at `src` (device) if it is missing.
cudaError_t build_layout(dspark_walk* h, Path which, const void* src) {
  cudaError_t e = cudaSuccess;
  void* s = const_cast<void*>(src);
  switch (which) {
    case Path::kMma:
      if (h->W2m || !h->mr_ok) return cudaSuccess;
      e = cudaMalloc(&h->W2m, (size_t)h->mr_wpc * h->mr_n_cta * sizeof(uint32_t));
      if (e == cudaSuccess)
        e = mma_resident_repack(s, h->W2m, h->V, h->mr_R, h->mr_S + h->mr_ST, h->mr_n_cta, false,
                                0);
      return e;
    case Path::kResident:
      if (h->W2p || h->res_max_B == 0) return cudaSuccess;
      e = cudaMalloc(&h->W2p, (size_t)h->res_wpc * h->res_n_cta * sizeof(uint32_t));
      if (e == cudaSuccess)
        e = resident_repack(s, h->W2p, h->V, h->res_R, h->res_RS, h->res_S + h->res_ST,
                            h->res_n_cta, false, 0);
      return e;
    case Path::kBatched:
      if (h->W2b) return cudaSuccess;
      e = cudaMalloc(&h->W2b, (size_t)h->bat_R * h->bat_n_cta * 512);
      if (e == cudaSuccess) e = batched_repack(s, h->W2b, h->V, h->bat_R, h->bat_n_cta, false, 0);
      return e;
    case Path::kStream:
      if (h->W2) return cudaSuccess;
      e = cudaMalloc(&h->W2, rowmajor_bytes(h));
      if (e == cudaSuccess) e = cudaMemcpy(h->W2, src, rowmajor_bytes(h), cudaMemcpyDeviceToDevice);
      return e;
  }
  return cudaErrorInvalidValue;
}

// Make sure a run of B requests finds its layout (built from the layouts the
// handle holds, through a temporary row-major copy).  Synchronises the device.
int ensure_layout(dspark_walk* h, int B) {
  const Path need = path_for(h, B);
  const bool have = (need == Path::kMma && h->W2m) || (need == Path::kResident && h->W2p) ||
                    (need == Path::kBatched && h->W2b) || (need == Path::kStream && h->W2);
  if (have) return DSPARK_OK;
  CUDA_TRY(cudaSetDevice(h->device));
  void* tmp = nullptr;
  const void* src = h->W2;
  if (!src) {
    CUDA_TRY(cudaMalloc(&tmp, rowmajor_bytes(h)));
    cudaError_t e = unpack_rowmajor(h, tmp);
    if (e != cudaSuccess) {
      cudaFree(tmp);
      return cuda_fail(e);
    }
    src = tmp;
  }
  cudaError_t e = build_layout(h, need, src);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (tmp) cudaFree(tmp);
  return e == cudaSuccess ? DSPARK_OK : cuda_fail(e);
}

// Every batch size a handle may run under its current settings.
int ensure_layouts(dspark_walk* h) {
  int rc = ensure_layout(h, 1);
  if (rc == DSPARK_OK) rc = ensure_layout(h, h->max_B);
  if (rc == DSPARK_OK && h->mr_max_B > 0 && h->mr_max_B < h->max_B)
    rc = ensure_layout(h, h->mr_max_B + 1);
  if (rc == DSPARK_OK && h->res_max_B > 0 && h->res_max_B < h->max_B)
    rc = ensure_layout(h, h->res_max_B + 1);
  return rc;
}

int64_t layout_bytes(const dspark_walk* h) {
  int64_t n = 0;
  if (h->W2) n += (int64_t)rowmajor_bytes(h);
  if (h->W2m) n += h->mr_wpc * h->mr_n_cta * 4;
  if (h->W2p) n += h->res_wpc * h->res_n_cta * 4;
  if (h->W2b) n += (int64_t)h->bat_R * h->bat_n_cta * 512;
  return n;
}

int launch_round(dspark_walk* h, const void* base, const int32_t* anchor, const float* temp,
                 uint64_t seed, int32_t* out_tokens, int B, int gamma, void* out_logits,
                 cudaStream_t stream) {
  WalkArgs a{};
  a.W1 = h->W1;
  a.W2 = h->W2;
  a.base = static_cast<const uint16_t*>(base);
  a.anchor = anchor;
  a.temperature = temp;
  a.out_tokens = out_tokens;
  a.out_logits = static_cast<uint16_t*>(out_logits);
  a.sync = h->sync;
  a.V = h->V;
  a.B = B;
  a.gamma = gamma;
  a.rows_per_cta = h->st_rpc;
  a.seed_lo = (uint32_t)seed;
  a.seed_hi = (uint32_t)(seed >> 32);
  a.seed_per_round = h->seed_per_round;
  a.sampler = h->sampler;
  a.timeout_ns = h->timeout_ns;
  a.skip_cta = h->skip_cta;
  const Path path = path_for(h, B);
  {
    const int n = path == Path::kMma        ? h->mr_n_cta
                  : path == Path::kResident ? h->res_n_cta
                  : path == Path::kBatched  ? h->bat_n_cta
                                            : h->st_n_cta;
    const int64_t need = (int64_t)n * (gamma + 1) * 8 * 8;
    a.trace = (h->trace && h->trace_bytes >= need) ? h->trace : nullptr;
    a.trace_global = h->trace_global;
  }

  a.out_state = h->out_state;
  a.cell = h->cell;
  a.cell_M = h->cell_M;
  a.cell_X = h->cell_X;
  a.cell_p = h->cell_p;
  a.cell_q = 1;
  // recurrent heads and the state output run on the tcgen05 resident kernel only
  if (cell_run(h) && path != Path::kResident) return DSPARK_EUNSUPPORTED;
  if (path == Path::kResident) {
    const int P = h->cell == DSPARK_CELL_GRU ? kCellP : kRank;   // recurrent rows
    a.cell_q = (P + h->res_n_cta - 1) / h->res_n_cta;
  }
  // the layout this run reads (set_kernel / set_cell build it when they
  // change the path; a handle always holds the layouts its settings need)
  const bool have = (path == Path::kMma && h->W2m) || (path == Path::kResident && h->W2p) ||
                    (path == Path::kBatched && h->W2b) || (path == Path::kStream && h->W2);
  if (!have) return DSPARK_EINTERNAL;

  if (path == Path::kBatched) {
    CUDA_TRY(batched_launch(a, h->W2b, h->bat_R, h->bat_n_cta, h->max_B, B,
                            232448 - 1024, stream));
    return DSPARK_OK;
  }

  if (path == Path::kMma || path == Path::kResident) {
    const bool mma = path == Path::kMma;
    ResidentArgs ra{};
    ra.w = a;
    ra.w.rows_per_cta = mma ? h->mr_R : h->res_R;
    ra.W2p = mma ? h->W2m : h->W2p;
    ra.R = mma ? h->mr_R : h->res_R;
    ra.S = mma ? h->mr_S : h->res_S;
    ra.ST = mma ? h->mr_ST : h->res_ST;
    ra.nslot = mma ? h->mr_nslot : h->res_nslot;
    ra.words_per_cta = mma ? h->mr_wpc : h->res_wpc;
    const uintptr_t bp = reinterpret_cast<uintptr_t>(base);
    ra.base_mode = (h->V % 8 == 0 && (bp & 15u) == 0) ? 16
                   : (h->V % 2 == 0 && (bp & 3u) == 0) ? 4 : 2;
    const void* rfn = mma ? mma_resident_kernel(h->mr_S, B <= 8 ? 1 : 2, h->mr_ST > 0)
                          : resident_kernel_for(h->res_RS, h->res_NT, cell_run(h));
    void* rargs[] = {&ra};
    CUDA_TRY(cudaLaunchCooperativeKernel(rfn, dim3(mma ? h->mr_n_cta : h->res_n_cta),
                                         dim3(resident_threads()), rargs,
                                         mma ? h->mr_smem : h->res_smem, stream));
    return DSPARK_OK;
  }

  // the streamed kernel scores one token per lane: the group sampler (8
  // consecutive tokens per group) is not available there
  if (h->sampler != DSPARK_SAMPLER_GUMBEL) return DSPARK_EUNSUPPORTED;
  const void* fn = stream_kernel_for(B);
  const size_t smem = stream_smem_bytes(B);  // <= the maximum set at create
  void* args[] = {&a};
  CUDA_TRY(cudaLaunchCooperativeKernel(fn, dim3(h->st_n_cta), dim3(stream_threads()), args,
                                       smem, stream));
  return DSPARK_OK;
}

// Device address of a host buffer the GPU can read in place (pinned memory,
// cudaHostAlloc or cudaHostRegister), or null.
const void* mapped_host(const void* p) {
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return pa.type == cudaMemoryTypeHost ? pa.devicePointer : nullptr;
}

// Base logits up to this size are read by the kernel straight from pinned
// host memory (each CTA fetches its rows one step ahead); larger ones are
// copied to the device first, where the kernel's reads run at HBM speed.
constexpr size_t kZeroCopyBaseMax = (size_t)16 << 20;

}  // namespace

extern "C" {

int dspark_walk_create(const void* W1, const void* W2, int64_t V, int r, int max_B,
                       int max_gamma, dspark_walk_t* out) {
  if (out) *out = nullptr;
  if (!W1 || !W2 || !out) return DSPARK_EINVAL;
  if (V < 1 || V >= ((int64_t)1 << 31)) return DSPARK_EINVAL;
  if (max_B < 1 || max_B > kMaxB || max_gamma < 1 || max_gamma > kMaxGamma) return DSPARK_EINVAL;
  if (r != kRank) return DSPARK_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(W1) & 15u) != 0 || (reinterpret_cast<uintptr_t>(W2) & 15u) != 0)
    return DSPARK_EINVAL;

  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  int major = 0, minor = 0, sms = 0, coop = 0;
  CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  CUDA_TRY(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  CUDA_TRY(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
  if (major != 10 || minor != 3 || !coop) return DSPARK_EUNSUPPORTED;

  dspark_walk* h = new (std::nothrow) dspark_walk();
  if (!h) return DSPARK_ENOMEM;
  h->device = dev;
  h->sm_count = sms;
  h->V = V;
  h->r = r;
  h->max_B = max_B;
  h->max_gamma = max_gamma;
  h->W1 = static_cast<const uint16_t*>(W1);

  int rc = DSPARK_OK;
  plan_mma(h);
  const bool resident = plan_resident(h);
  plan_batched(h);
  size_t count_off, key_off, slot_off, total;
  const int slot_B = max_B < 16 ? max_B : 16;
  const int slot_stride = (sms + 15) / 16 * 16;
  sync_layout(max_gamma, max_B, slot_B, slot_stride, &count_off, &key_off, &slot_off, &total);
  cudaError_t e = cudaMalloc(&h->sync_mem, total);
  if (e == cudaSuccess) e = cudaMemset(h->sync_mem, 0, total);
  if (e == cudaSuccess) {
    uint8_t* base = static_cast<uint8_t*>(h->sync_mem);
    h->sync.hdr = reinterpret_cast<SyncHeader*>(base);
    h->sync.count = reinterpret_cast<uint32_t*>(base + count_off);
    h->sync.key = reinterpret_cast<unsigned long long*>(base + key_off);
    h->sync.max_gamma = max_gamma;
    h->sync.max_B = max_B;
    h->sync.slot = reinterpret_cast<unsigned long long*>(base + slot_off);
    h->sync.slot_B = slot_B;
    h->sync.slot_stride = slot_stride;
  }
  if (e != cudaSuccess) rc = cuda_fail(e);
  if (rc == DSPARK_OK) {
    plan_stream(h);
    // every instantiation may use the shared memory of max_B, and one CTA
    // per SM must fit.  A kernel's shared-memory limit is one setting for the
    // whole process, shared by every handle (and the allocation-free entry):
    // it is raised to what the largest batch needs, never lowered to this
    // handle's need.
    const size_t smem = stream_smem_bytes(max_B);
    for (int b = 1; b <= 8 && rc == DSPARK_OK; b *= 2) {
      int per_sm = 0;
      const void* fn = stream_kernel_for(b);
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)stream_smem_bytes(kMaxB));
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, stream_threads(), smem);
      if (e != cudaSuccess) rc = cuda_fail(e);
      else if (per_sm < 1) rc = DSPARK_EUNSUPPORTED;
    }
    if (rc == DSPARK_OK) {
      int per_sm = 0;
      e = cudaFuncSetAttribute(batched_kernel(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               232448 - 1024);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, batched_kernel(),
                                                          batched_threads(), 232448 - 1024);
      if (e != cudaSuccess) rc = cuda_fail(e);
      else if (per_sm != 1) rc = DSPARK_EUNSUPPORTED;
    }
    if (rc == DSPARK_OK && resident) {
      int per_sm = 0;
      const void* fn = resident_kernel_for(h->res_RS, h->res_NT, false);
      const void* fn_cell = resident_kernel_for(h->res_RS, h->res_NT, true);
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBudget);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn_cell, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemBudget);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, resident_threads(),
                                                          h->res_smem);
      // exactly one CTA per SM: two would contend for the whole tensor memory
      if (e != cudaSuccess || per_sm != 1) {
        // the resident kernel cannot run here: every run streams instead
        cudaGetLastError();
        h->res_max_B = 0;
      }
    }
    if (rc == DSPARK_OK && h->mr_ok) {
      int per_sm = 0;
      for (int s = 0; s <= 24 && e == cudaSuccess; s += 8)
        for (int nt = 1; nt <= 2 && e == cudaSuccess; ++nt)
          for (int str = 0; str <= (s <= 16 ? 1 : 0) && e == cudaSuccess; ++str)
            e = cudaFuncSetAttribute(mma_resident_kernel(s, nt, str != 0),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBudget);
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, mma_resident_kernel(h->mr_S, h->mr_max_B > 8 ? 2 : 1, h->mr_ST > 0),
            resident_threads(), h->mr_smem);
      if (e != cudaSuccess || per_sm != 1) {
        cudaGetLastError();
        h->mr_ok = false;
        h->mr_max_B = 0;
      }
    }
    plan_stream(h);
  }
  // the layouts the runs of this handle can take, each repacked from the
  // caller's W2 (no row-major copy is kept)
  if (rc == DSPARK_OK) {
    const Path paths[] = {path_for(h, 1), path_for(h, max_B),
                          path_for(h, h->mr_max_B > 0 && h->mr_max_B < max_B ? h->mr_max_B + 1 : 1),
                          path_for(h, h->res_max_B > 0 && h->res_max_B < max_B ? h->res_max_B + 1
                                                                                 : 1)};
    for (const Path pth : paths) {
      e = build_layout(h, pth, W2);
      if (e != cudaSuccess) break;
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) rc = cuda_fail(e);
  }
  if (rc != DSPARK_OK) {
    dspark_walk_destroy(h);
    return rc;
  }
  *out = h;
  return DSPARK_OK;
}

int dspark_walk_run(dspark_walk_t h, const void* base_logits, const int32_t* anchor,
                    const float* temperature, uint64_t seed, int32_t* out_tokens, int B,
                    int gamma, void* out_logits, void* stream) {
  if (!h || !base_logits || !anchor || !temperature || !out_tokens) return DSPARK_EINVAL;
  if (B < 1 || B > h->max_B || gamma < 1 || gamma > h->max_gamma) return DSPARK_EINVAL;
  return launch_round(h, base_logits, anchor, temperature, seed, out_tokens, B, gamma,
                      out_logits, static_cast<cudaStream_t>(stream));
}

int dspark_walk_run_host(dspark_walk_t h, const void* base_logits_host,
                         const int32_t* anchor_host, const float* temperature_host,
                         uint64_t seed, int32_t* out_tokens_host, int B, int gamma,
                         void* out_logits_host, void* stream) {
  if (!h || !base_logits_host || !anchor_host || !temperature_host || !out_tokens_host)
    return DSPARK_EINVAL;
  if (B < 1 || B > h->max_B || gamma < 1 || gamma > h->max_gamma) return DSPARK_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // device staging: base | logits | tokens (each used only when the host
  // buffer cannot be read or written in place)
  const size_t nlog = (size_t)h->max_B * h->max_gamma * (size_t)h->V;
  const size_t off_logits = round_up(nlog * 2, 256);
  const size_t off_tok = off_logits + round_up(nlog * 2, 256);
  const size_t need = off_tok + round_up((size_t)h->max_B * h->max_gamma * 4, 256);
  if (h->stage_bytes < need) {
    if (h->stage) cudaFree(h->stage);
    h->stage = nullptr;
    h->stage_bytes = 0;
    CUDA_TRY(cudaMalloc(&h->stage, need));
    h->stage_bytes = need;
  }
  // pinned, mapped host block {anchor[max_B], temperature[max_B], status}
  const size_t small = (size_t)h->max_B * 8;
  if (!h->hstage) CUDA_TRY(cudaHostAlloc(&h->hstage, small + 16, cudaHostAllocMapped));
  uint8_t* st = static_cast<uint8_t*>(h->stage);
  uint8_t* hs = static_cast<uint8_t*>(h->hstage);
  void* hs_dev = nullptr;
  CUDA_TRY(cudaHostGetDevicePointer(&hs_dev, h->hstage, 0));
  // the previous call synchronised its stream, so the block is free
  memcpy(hs, anchor_host, (size_t)B * 4);
  memcpy(hs + (size_t)h->max_B * 4, temperature_host, (size_t)B * 4);
  int32_t* hstatus = reinterpret_cast<int32_t*>(hs + small);
  const size_t nb = (size_t)B * gamma * (size_t)h->V * 2;
  const void* base_dev = nb <= kZeroCopyBaseMax ? mapped_host(base_logits_host) : nullptr;
  if (!base_dev) {
    CUDA_TRY(cudaMemcpyAsync(st, base_logits_host, nb, cudaMemcpyHostToDevice, s));
    base_dev = st;
  }
  int32_t* tok_dev = static_cast<int32_t*>(const_cast<void*>(mapped_host(out_tokens_host)));
  const bool tok_copy = tok_dev == nullptr;
  if (tok_copy) tok_dev = reinterpret_cast<int32_t*>(st + off_tok);
  const uint8_t* hsd = static_cast<const uint8_t*>(hs_dev);
  int rc = launch_round(h, base_dev, reinterpret_cast<const int32_t*>(hsd),
                        reinterpret_cast<const float*>(hsd + (size_t)h->max_B * 4), seed, tok_dev,
                        B, gamma, out_logits_host ? st + off_logits : nullptr, s);
  if (rc != DSPARK_OK) return rc;
  if (tok_copy)
    CUDA_TRY(cudaMemcpyAsync(out_tokens_host, tok_dev, (size_t)B * gamma * 4,
                             cudaMemcpyDeviceToHost, s));
  if (out_logits_host)
    CUDA_TRY(cudaMemcpyAsync(out_logits_host, st + off_logits, nb, cudaMemcpyDeviceToHost, s));
  // the round's status rides on the same stream: one synchronisation in all
  CUDA_TRY(cudaMemcpyAsync(hstatus, &h->sync.hdr->status, sizeof(int32_t),
                           cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  const int32_t code = *hstatus;
  if (code != 0) {                                   // clear it for the next run
    const int32_t zero = 0;
    CUDA_TRY(cudaMemcpy(&h->sync.hdr->status, &zero, sizeof zero, cudaMemcpyHostToDevice));
  }
  return code;
}

int dspark_walk_status(dspark_walk_t h, void* stream) {
  if (!h) return DSPARK_EINVAL;
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int32_t st = 0;
  CUDA_TRY(cudaMemcpy(&st, &h->sync.hdr->status, sizeof st, cudaMemcpyDeviceToHost));
  if (st != 0) {
    const int32_t zero = 0;
    CUDA_TRY(cudaMemcpy(&h->sync.hdr->status, &zero, sizeof zero, cudaMemcpyHostToDevice));
  }
  return st;
}

int dspark_walk_get_plan(dspark_walk_t h, struct dspark_walk_plan* p) {
  if (!h || !p) return DSPARK_EINVAL;
  *p = h->plan;
  p->weight_bytes = layout_bytes(h);
  return DSPARK_OK;
}

int dspark_walk_set_limits(dspark_walk_t h, int64_t timeout_ns, int skip_cta) {
  if (!h || timeout_ns < 1000 || skip_cta < -1) return DSPARK_EINVAL;
  h->timeout_ns = timeout_ns;
  h->skip_cta = skip_cta;
  return DSPARK_OK;
}

int dspark_walk_set_trace(dspark_walk_t h, void* device_buffer, int64_t bytes) {
  if (!h || bytes < 0 || (device_buffer == nullptr && bytes != 0)) return DSPARK_EINVAL;
  h->trace = static_cast<unsigned long long*>(device_buffer);
  h->trace_bytes = bytes;
  return DSPARK_OK;
}

int dspark_walk_set_trace_clock(dspark_walk_t h, int clock) {
  if (!h || (clock != DSPARK_TRACE_SM_CLOCK && clock != DSPARK_TRACE_GLOBAL_TIMER))
    return DSPARK_EINVAL;
  h->trace_global = clock == DSPARK_TRACE_GLOBAL_TIMER ? 1 : 0;
  return DSPARK_OK;
}

int dspark_walk_set_kernel(dspark_walk_t h, int kernel) {
  if (!h) return DSPARK_EINVAL;
  const bool r0 = h->use_resident, b0 = h->use_batched;
  if (kernel == DSPARK_KERNEL_STREAM) {
    h->use_resident = false;
    h->use_batched = false;
  } else if (kernel == DSPARK_KERNEL_RESIDENT) {
    if (h->res_max_B == 0 && !h->mr_ok) return DSPARK_EUNSUPPORTED;
    h->use_resident = true;
    h->use_batched = true;
  } else if (kernel == DSPARK_KERNEL_BATCHED) {
    h->use_resident = false;
    h->use_batched = true;
  } else {
    return DSPARK_EINVAL;
  }
  const int rc = ensure_layouts(h);
  if (rc != DSPARK_OK) {
    h->use_resident = r0;
    h->use_batched = b0;
  }
  return rc;
}

int dspark_walk_set_seed_mode(dspark_walk_t h, int mode) {
  if (!h || (mode != DSPARK_SEED_FIXED && mode != DSPARK_SEED_PER_ROUND)) return DSPARK_EINVAL;
  h->seed_per_round = mode == DSPARK_SEED_PER_ROUND ? 1 : 0;
  return DSPARK_OK;
}

int dspark_walk_set_sampler(dspark_walk_t h, int sampler) {
  if (!h || (sampler != DSPARK_SAMPLER_GUMBEL && sampler != DSPARK_SAMPLER_GROUP))
    return DSPARK_EINVAL;
  h->sampler = sampler;
  return DSPARK_OK;
}

int dspark_walk_set_cell(dspark_walk_t h, int cell, const void* M, const void* X) {
  if (!h) return DSPARK_EINVAL;
  if (cell == DSPARK_CELL_MARKOV) {
    h->cell = cell;
    h->cell_M = h->cell_X = nullptr;
    return DSPARK_OK;
  }
  if ((cell != DSPARK_CELL_GATED && cell != DSPARK_CELL_RNN && cell != DSPARK_CELL_GRU) || !M ||
      (reinterpret_cast<uintptr_t>(M) & 15u) != 0)
    return DSPARK_EINVAL;
  if (cell == DSPARK_CELL_GRU && (!X || (reinterpret_cast<uintptr_t>(X) & 15u) != 0))
    return DSPARK_EINVAL;
  if (h->res_max_B == 0) return DSPARK_EUNSUPPORTED;   // no resident layout to run on
  if (!h->cell_p) {
    CUDA_TRY(cudaSetDevice(h->device));
    CUDA_TRY(cudaMalloc(&h->cell_p, (size_t)h->max_gamma * 16 * kCellP * sizeof(float)));
  }
  const int cell0 = h->cell;
  h->cell = cell;
  const int rc = ensure_layouts(h);
  if (rc != DSPARK_OK) {
    h->cell = cell0;
    return rc;
  }
  h->cell_M = static_cast<const uint16_t*>(M);
  h->cell_X = cell == DSPARK_CELL_GRU ? static_cast<const uint16_t*>(X) : nullptr;
  return DSPARK_OK;
}

int dspark_walk_set_state_output(dspark_walk_t h, void* out_state) {
  if (!h || (reinterpret_cast<uintptr_t>(out_state) & 1u) != 0) return DSPARK_EINVAL;
  uint16_t* prev = h->out_state;
  h->out_state = static_cast<uint16_t*>(out_state);
  if (out_state && h->res_max_B > 0) {
    const int rc = ensure_layouts(h);
    if (rc != DSPARK_OK) {
      h->out_state = prev;
      return rc;
    }
  }
  return DSPARK_OK;
}

int dspark_walk_round(dspark_walk_t h, void* stream, uint64_t* round) {
  if (!h || !round) return DSPARK_EINVAL;
  CUDA_TRY(cudaSetDevice(h->device));
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  uint32_t r = 0;
  CUDA_TRY(cudaMemcpy(&r, &h->sync.hdr->round, sizeof(r), cudaMemcpyDeviceToHost));
  *round = r;
  return DSPARK_OK;
}

int dspark_walk_gumbel_noise(const uint32_t* bits, float* noise, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && (!bits || !noise))) return DSPARK_EINVAL;
  if (n == 0) return DSPARK_OK;
  CUDA_TRY(gumbel_noise_launch(bits, noise, n, static_cast<cudaStream_t>(stream)));
  return DSPARK_OK;
}

const char* dspark_walk_strerror(int code) {
  switch (code) {
    case DSPARK_OK: return "ok";
    case DSPARK_EINVAL: return "invalid argument";
    case DSPARK_ENOMEM: return "out of device memory";
    case DSPARK_ECUDA: return "CUDA runtime error";
    case DSPARK_ETIMEOUT: return "cross-CTA rendezvous timed out";
    case DSPARK_EANCHOR: return "anchor token outside [0, V)";
    case DSPARK_EUNSUPPORTED: return "unsupported rank or device (needs r = 256 on sm_103)";
    case DSPARK_ETEMP: return "temperature negative or not finite";
    case DSPARK_EINTERNAL: return "device-side consistency check failed";
    case DSPARK_ELIMIT:
      return "batch or walk length above the allocation-free entry point's maximum (B <= 64, "
             "gamma <= 16)";
    default: return "unknown status";
  }
}

int dspark_walk_destroy(dspark_walk_t h) {
  if (!h) return DSPARK_EINVAL;
  int rc = DSPARK_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) rc = DSPARK_ECUDA;
  if (h->W2) cudaFree(h->W2);
  if (h->W2p) cudaFree(h->W2p);
  if (h->W2b) cudaFree(h->W2b);
  if (h->W2m) cudaFree(h->W2m);
  if (h->sync_mem) cudaFree(h->sync_mem);
  if (h->stage) cudaFree(h->stage);
  if (h->hstage) cudaFreeHost(h->hstage);
  if (h->cell_p) cudaFree(h->cell_p);
  delete h;
  return rc;
}

}  // extern "C"
