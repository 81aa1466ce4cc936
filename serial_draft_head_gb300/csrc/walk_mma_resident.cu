// walk_mma_resident.cu -- the persistent walk with W2 held on chip for the
// whole round, every tier read by mma.sync: "Keeping the Draft Walk on Chip:
// One Launch for DSpark's Markov Head", sections "The idea: make the walk
// resident" (one CTA per SM, one launch per round, each CTA loads its slice of
// rows once and runs all gamma steps, only token ids cross between steps) and
// "B200: the bf16 table fits on chip" (the table split over tensor memory,
// shared memory and registers; fp32 accumulation, bias rounded to bf16, then
// the sum rounded to bf16; request n is column n of the MMA's N operand).
//
// The pages' B200 kernel reads its tensor-memory rows with tcgen05.mma.  At one
// request the MMA's N operand is nearly empty, so what bounds a step is how fast
// each tier hands rows to the tensor cores, plus the fixed costs around the
// MMAs.  On GB300 a tcgen05.mma costs ~45 cycles to issue from one thread, its
// accumulators take tensor-memory columns, and its results need an extra
// completion wait and read-out per step.  Here tensor memory instead holds W2
// rows already laid out as mma.sync A fragments, in all 512 columns, and each
// warp streams its 32 KB share into registers with tcgen05.ld (~384 B per
// cycle per SM) one k-tile pair ahead of the mma.sync that consume them.  All
// three tiers then run as independent accumulation chains of one k loop.
//
// Per CTA (256 threads, 8 warps) the R rows of its shard are placed as
//   rows [0, 512)            tensor memory: warp w holds strips 4w .. 4w + 3
//                            (16 rows each) in lanes 32 (w % 4) .. + 31,
//                            columns 256 (w / 4) .. + 255;
//   rows [512, 640)          registers: one 16-row strip per warp;
//   rows [640, 640 + 128 NS) shared memory: NS = 0..3 strips per warp (the
//                            same count in every warp), read by ldmatrix;
//   rows [640 + 128 NS, R)   (shards past 1,024 rows, "V = 248,320: 62% on
//                            chip, the rest streamed") streamed every step:
//                            NS <= 2, and the remaining strips come from L2
//                            through a ring of 2 or 3 shared-memory slots of
//                            64 KB, one strip of every warp per slot (one
//                            bulk copy, one mbarrier); the last warp done
//                            with a slot refills it, so the next step's
//                            first slots load during the rendezvous.
// Requests: B <= 16 (one or two mma.sync n-tiles).  Larger batches and the
// recurrent heads run the other kernels.
//
// Epilogue: when every request of the round is greedy and no logits are
// written, each thread turns its accumulators straight into 32-bit keys {bf16
// logit order bits : 16, inverted local row : 16} and the maxima go through
// two warp and one CTA reduction; otherwise the logits are written into the
// shared base buffer and the common key pass scores them (Gumbel-max, the
// group sampler, the logits copy).
#include "resident_pass.cuh"
#include "tc_ptx.cuh"
#include "walk_common.cuh"
#include "walk_kernels.h"

namespace dspark {

namespace {

constexpr int kMrWarps = kResWarps;                   // 8
constexpr int kTmStrips = 4;                          // tensor-memory strips per warp
constexpr int kTmRows = kMrWarps * kTmStrips * 16;    // 512
constexpr int kRfRows = kMrWarps * 16;                // 128
constexpr int kMrFixedRows = kTmRows + kRfRows;       // 640
constexpr int kMrSmax = 3;                            // shared strips per warp, at most
constexpr int kMrMaxRows = kMrFixedRows + kMrSmax * kMrWarps * 16;   // 1024
constexpr int kMrMaxB = 16;
constexpr int kMrMaxCtas = 192;                     // CTAs whose slots one poll reads
constexpr int kTmWordsPerWarp = 32 * 256;             // 32 lanes x 256 columns
constexpr int kTmWords = kMrWarps * kTmWordsPerWarp;  // 256 KB
constexpr int kMrRfWords = kMrWarps * 16 * 32 * 4;    // 64 KB
constexpr int kMbarSmem = 0;
constexpr unsigned long long kKey50Mask = (1ull << 50) - 1ull;
constexpr int kRingSlotBytes = kMrWarps * kSmemStripBytes;   // 64 KB: a strip of every warp
constexpr int kMrMaxSlots = 4;                        // ring slots, at most
constexpr int kStreamGroup = 4;                       // streamed strips scored together
// the ring's control block after the slots: full mbarriers [kMrMaxSlots],
// warps still reading each slot [kMrMaxSlots], items issued, items freed
constexpr int kRingCtlBytes = 128;                    // keeps U 16-byte aligned

// Local row of the first row of strip st of warp w: st 0..3 tensor memory,
// 4 the register strip, 5.. shared memory (the j-th shared strip of the warp
// being strip w + 8 j of the shared tier).  Increasing st, increasing rows:
// the fused epilogue's running argmax relies on it for its ties.
__device__ __forceinline__ int strip_row0(int st, int w) {
  if (st < kTmStrips) return 16 * (kTmStrips * w + st);
  if (st == kTmStrips) return kTmRows + 16 * w;
  return kMrFixedRows + 16 * (w + kMrWarps * (st - 1 - kTmStrips));
}

// Order bits of two bf16 values packed in a word (-0 folded onto +0): larger
// value, larger bits, as the resident key pass forms them.
__device__ __forceinline__ uint32_t bf16_order(uint32_t x) {
  x = x == 0x8000u ? 0u : x;
  return (x & 0x8000u) ? (~x & 0xFFFFu) : (x | 0x8000u);
}

__device__ __forceinline__ uint32_t max_u32(uint32_t a, uint32_t b) { return a > b ? a : b; }

// Bits of a bf16 pair (two logits), as __nv_bfloat162.
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t x) {
  return *reinterpret_cast<const __nv_bfloat162*>(&x);
}
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 x) {
  return *reinterpret_cast<const uint32_t*>(&x);
}

// Running argmax of two independent streams of bf16 logits packed in one
// word (each half its own stream): where a half of `l` is greater than the
// same half of `best`, it replaces it and its row (a half of `rows`) replaces
// the kept row.  Rows come in increasing order, so the strict comparison
// keeps the smallest row among equal logits; -0 and +0 compare equal.
__device__ __forceinline__ void argmax2(uint32_t l, uint32_t rows, uint32_t& best,
                                        uint32_t& best_rows) {
  const uint32_t m = __hgt2_mask(as_bf2(l), as_bf2(best));
  best = (l & m) | (best & ~m);
  best_rows = (rows & m) | (best_rows & ~m);
}

// {bf16 order bits : 16, inverted local row : 16} of a bf16 logit and its
// row (-0 folded onto +0).
__device__ __forceinline__ uint32_t key32(uint32_t lb, uint32_t row) {
  return (bf16_order(lb & 0xFFFFu) << 16) | (0xFFFFu - (row & 0xFFFFu));
}

// The fused epilogue of a greedy round without logits out, for one warp:
// each request's best key over the warp's NST strips, 32-bit {bf16 logit
// order bits : 16, inverted local row : 16}, into wkey[b].
// Lane (g, t4) holds rows g and g + 8 of columns 2 t4 and 2 t4 + 1 (requests)
// of every strip.  With B <= 8 / G requests only the lanes t4 < 4 / G hold
// results, so they are first spread over the G lane groups: lane (g, t4)
// takes strips s = part (mod G), part = t4 / (4 / G), from lane (g, t4 mod
// (4 / G)).  Every lane then scores NST / G strips, two logits per
// instruction: the two bias roundings in one bf16x2 conversion, the base add
// as one correctly rounded bf16x2 addition (for bf16 operands the same value
// as bf16(fp32 sum), whose fp32 sum is exact whenever it could matter), and a
// packed running argmax (argmax2).  The pairs are the two requests of a row,
// or, with one request, rows g and g + 8.  Rows past the shard's end score
// -inf.  Then a max over the lanes that hold the same request.  accs[s] is
// strip st0 + s of the warp; only the first nst of them are real; MERGE keeps
// the larger of wkey[b] and the new key (strips scored in several calls).
template <int NST, int G, int NT, bool MERGE = false>
__device__ __forceinline__ void fast_keys(const float (&accs)[NST][NT][4], int nt,
                                          const uint16_t* base_s, int R, int B, int nv, int warp,
                                          int lane, uint32_t* wkey, int st0 = 0, int nst = NST) {
  constexpr int NJ = (NST + G - 1) / G;          // strips per lane
  constexpr int SRC = 4 / G;                     // lanes per row group holding results
  constexpr uint32_t kNegInf2 = 0xFF80FF80u;
  const int g = lane >> 2, t4 = lane & 3;
  const int src = t4 % SRC, part = t4 / SRC;
  const int bq = 8 * nt;                         // requests of this n-tile: bq + column
  B -= bq;
  wkey += bq;
  float v[NJ][4];
#pragma unroll
  for (int s = 0; s < NST; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a_ = accs[s][nt][e];
      const float x = G > 1 ? __shfl_sync(0xFFFFFFFFu, a_, (lane & ~3) | src) : a_;
      if (G == 1 || s % G == part) v[s / G][e] = x;
    }
  int rr[NJ], rl[NJ][2];              // rows; the rows the base loads read (kept below R)
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int s = part + G * j;
    rr[j] = s < nst ? strip_row0(st0 + s, warp) + g : 0;
    rl[j][0] = rr[j] < R ? rr[j] : R - 1;            // a padding strip's rows lie past R
    rl[j][1] = rr[j] + 8 < R ? rr[j] + 8 : R - 1;
  }
  uint32_t best = kNegInf2, brow = 0xFFFFFFFFu;
  if (G == 4 && B == 1) {
    // pairs = rows (g, g + 8) of request 0
    uint32_t bb[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      bb[j] = (uint32_t)base_s[rl[j][0]] | ((uint32_t)base_s[rl[j][1]] << 16);
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t bias = bf2_bits(__floats2bfloat162_rn(v[j][0], v[j][2]));
      uint32_t l = bf2_bits(__hadd2(as_bf2(bb[j]), as_bf2(bias)));
      const bool ok = part + G * j < nst;
      const uint32_t lo_ok = ok && rr[j] < nv ? 0u : 0x0000FFFFu;
      const uint32_t hi_ok = ok && rr[j] + 8 < nv ? 0u : 0xFFFF0000u;
      l = (l & ~(lo_ok | hi_ok)) | (kNegInf2 & (lo_ok | hi_ok));
      argmax2(l, (uint32_t)rr[j] | ((uint32_t)(rr[j] + 8) << 16), best, brow);
    }
    const uint32_t k0 = key32(best, brow), k1 = key32(best >> 16, brow >> 16);
    uint32_t kb = max_u32(k0, k1);
    if (best == kNegInf2 && k0 == k1) kb = 0u;    // no valid row at all
    kb = ptx::redux_max_u32(kb);
    if (lane == 0) wkey[0] = MERGE ? max_u32(wkey[0], kb) : kb;
    return;
  }
  // pairs = requests (2 src, 2 src + 1) of one row
  const int b0 = 2 * src < B ? 2 * src : 0, b1 = 2 * src + 1 < B ? 2 * src + 1 : 0;
  const uint16_t* bs0 = base_s + (size_t)(bq + b0) * R;
  const uint16_t* bs1 = base_s + (size_t)(bq + b1) * R;
  uint32_t bb[NJ][2];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      bb[j][h] = (uint32_t)bs0[rl[j][h]] | ((uint32_t)bs1[rl[j][h]] << 16);
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t bias = bf2_bits(__floats2bfloat162_rn(v[j][2 * h], v[j][2 * h + 1]));
      uint32_t l = bf2_bits(__hadd2(as_bf2(bb[j][h]), as_bf2(bias)));
      const int row = rr[j] + 8 * h;
      if (!(part + G * j < nst && row < nv)) l = kNegInf2;
      argmax2(l, (uint32_t)row * 0x10001u, best, brow);
    }
  uint32_t kb[2] = {key32(best, brow), key32(best >> 16, brow >> 16)};
  // lanes with the same src hold the same two requests: reduce over g and part
  if constexpr (SRC == 1) {
#pragma unroll
    for (int q = 0; q < 2; ++q) kb[q] = ptx::redux_max_u32(kb[q]);
  } else if constexpr (SRC <= 4) {        // one masked maximum per src
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t r = 0u;
#pragma unroll
      for (int sv = 0; sv < SRC; ++sv) {
        const uint32_t m = ptx::redux_max_u32(src == sv ? kb[q] : 0u);
        r = src == sv ? m : r;
      }
      kb[q] = r;
    }
  } else {
#pragma unroll
    for (int o = SRC; o < 32; o <<= 1)
#pragma unroll
      for (int q = 0; q < 2; ++q) kb[q] = max_u32(kb[q], __shfl_xor_sync(0xFFFFFFFFu, kb[q], o));
  }
  if (g == 0 && part == 0)
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (2 * src + q < B) wkey[2 * src + q] = MERGE ? max_u32(wkey[2 * src + q], kb[q]) : kb[q];
}

template <int NS, int NT, bool STR>
__global__ void __launch_bounds__(kResThreads, 1) walk_mma_kernel(const ResidentArgs ra) {
  constexpr int NST = 1 + kTmStrips + NS;
  const WalkArgs& a = ra.w;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* smem_w2 = smem;
  uint8_t* ring = smem + (size_t)ra.S * kSmemStripBytes;   // STR: nslot slots of 64 KB
  const int nslot = STR ? ra.nslot : 0;
  uint8_t* ring_ctl = ring + (size_t)nslot * kRingSlotBytes;
  uint64_t* ring_bar = reinterpret_cast<uint64_t*>(ring_ctl);
  int* ring_left = reinterpret_cast<int*>(ring_ctl + 8 * kMrMaxSlots);
  int* ring_sent = ring_left + kMrMaxSlots;            // items issued so far
  int* ring_freed = ring_sent + 1;                     // items every warp has read
  uint8_t* U = ring_ctl + (STR ? kRingCtlBytes : 0);
  uint16_t* base_s = reinterpret_cast<uint16_t*>(U + 16 * 512);
  __shared__ __align__(8) uint64_t mbar[1];
  __shared__ unsigned long long group_best[16][kResWarps];
  __shared__ uint32_t warp_key[kMrWarps][kMrMaxB];
  __shared__ float temp_s[16];
  __shared__ int32_t tok_s[16];
  __shared__ uint32_t tmem_base_s;
  __shared__ int flag_s;
  __shared__ int fast_s;
  __shared__ int abort_s;
  __shared__ uint32_t round_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int cta = blockIdx.x;
  const int n_cta = gridDim.x;
  const int64_t row0 = (int64_t)cta * ra.R;
  const int nv = (int)((a.V - row0) < ra.R ? (a.V - row0) : ra.R);  // valid rows (>= 1)
  const uint32_t* gw = ra.W2p + (size_t)cta * (size_t)ra.words_per_cta;

  trace_stamp(a, a.gamma, 3);          // the CTA's first instruction
  const int bad = check_inputs(a, &flag_s);
  if (bad != 0) {
    if (cta == 0) {
      if (threadIdx.x == 0) set_status(a.sync.hdr, bad);
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    }
    return;
  }

  // ------------------------------------------------------------- entry ----
  trace_stamp(a, a.gamma, 0);
  if (threadIdx.x == 0) {
    round_s = *reinterpret_cast<volatile uint32_t*>(&a.sync.hdr->round);
    abort_s = 0;
    ptx::mbar_init(&mbar[kMbarSmem], 1);
    if constexpr (STR) {
      for (int i = 0; i < nslot; ++i) {
        ptx::mbar_init(&ring_bar[i], 1);
        ring_left[i] = kMrWarps;
      }
      *ring_sent = 0;
      *ring_freed = 0;
    }
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base_s, 512);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x < 16) {
    temp_s[threadIdx.x] = threadIdx.x < a.B ? a.temperature[threadIdx.x] : 0.0f;
    tok_s[threadIdx.x] = threadIdx.x < a.B ? a.anchor[threadIdx.x] : 0;
  }
  for (int i = threadIdx.x; i < 16 * 512 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(U)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  if (threadIdx.x == 0) {      // every request greedy and no logits out: fused keys
    int f = a.out_logits == nullptr ? 1 : 0;
    for (int b = 0; b < a.B; ++b) f = (temp_s[b] == 0.0f) ? f : 0;
    fast_s = f;
  }

  // this CTA's slots of the other parity start empty for the next round, and
  // so do that parity's arrival counts
  clear_own_slots(a.sync, round_s & 1u);
  if (cta == 0) clear_other_parity(a.sync, round_s & 1u);

  // The shard is read from memory once per round, so its loads carry an L2
  // evict-first policy: when the round starts on an L2 full of other data
  // (a drafter's forward pass runs between two walks, so it usually does),
  // the shard's own lines are replaced before that data, and lines that
  // would have to be written back first stay.  (Back-to-back rounds then
  // find less of the shard in L2.)  The streamed tier is the other way round:
  // evict-last, read every step.
  const uint64_t pol_first = ptx::policy_evict_first();

  // shared-memory tier: bulk copies straight to its final place
  const uint64_t t_entry = globaltimer_ns();
  if (threadIdx.x == 0 && ra.S > 0) {
    const uint32_t bytes = (uint32_t)ra.S * kSmemStripBytes;
    ptx::mbar_expect_tx(&mbar[kMbarSmem], bytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(gw + kTmWords + kMrRfWords);
    for (uint32_t off = 0; off < bytes; off += 32768u) {
      const uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
      ptx::bulk_g2s_hint(smem_w2 + off, src + off, n, &mbar[kMbarSmem], pol_first);
    }
  }

  // streamed tier: the CTA's ST strips past the shared tier, ST / 8 per warp
  // (warp w's i-th is shared-tier strip S + 8 i + w, rows 640 + 16 (S + 8 i +
  // w)), go through a ring of nslot 64 KB slots every step: item n of the
  // round (step n / nt2, i = n % nt2) is the i-th streamed strip of every
  // warp, one contiguous bulk copy, warp w's strip at w * 8 KB.  The last
  // warp done with a slot refills it with item n + nslot, so the next step's
  // first items load while this step finishes.  L2 keeps these rows
  // (evict-last): they are read every step.
  const int nt2 = STR ? ra.ST / kMrWarps : 0;        // streamed strips per warp
  const int ring_total = a.gamma * nt2;              // items per round
  const uint64_t pol_stream = ptx::policy_evict_last();
  auto ring_issue = [&](int n) {                     // one thread
    const uint8_t* src = reinterpret_cast<const uint8_t*>(gw + kTmWords + kMrRfWords) +
                         (size_t)(ra.S + kMrWarps * (n % nt2)) * kSmemStripBytes;
    uint64_t* bar = &ring_bar[n % nslot];
    ptx::mbar_expect_tx(bar, kRingSlotBytes);
    ptx::bulk_g2s_hint(ring + (size_t)(n % nslot) * kRingSlotBytes, src, kRingSlotBytes, bar,
                       pol_stream);
  };
  if (STR && threadIdx.x == 0) {
    const int pre = ring_total < nslot ? ring_total : nslot;
    for (int n = 0; n < pre; ++n) ring_issue(n);
    *ring_sent = pre;
  }

  // step 0's base rows: asynchronous copies, in flight during the loads below
  prefetch_base(ra, 0, row0, nv, base_s);

  // register tier and tensor-memory tier: global -> registers (-> tcgen05.st).
  // Warp w's tensor-memory block is 8 chunks of 32 columns; lane l's 32 words
  // of chunk p sit at [w][p][m][l][4], m = 0..7 (512 contiguous bytes per load).
  const uint32_t tq = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tcol = 256u * (uint32_t)(warp >> 2);
  const uint32_t tm_addr = tmem + tq + tcol;
  uint32_t wr[16][4];                  // register tier: this warp's strip as A fragments
  {
    const uint4* rsrc = reinterpret_cast<const uint4*>(gw + kTmWords) + (size_t)warp * 16 * 32 + lane;
    const uint4* tsrc = reinterpret_cast<const uint4*>(gw) + (size_t)warp * (kTmWordsPerWarp / 4) + lane;
    uint32_t v0[32], v1[32];
    auto load_chunk = [&](int p, uint32_t (&v)[32]) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint4 x = ptx::ldg_nc_na_hint(tsrc + (p * 8 + m) * 32, pol_first);
        v[4 * m + 0] = x.x;
        v[4 * m + 1] = x.y;
        v[4 * m + 2] = x.z;
        v[4 * m + 3] = x.w;
      }
    };
    auto store_chunk = [&](int p, uint32_t (&v)[32]) { ptx::tmem_st32(tm_addr + 32 * p, v); };
    load_chunk(0, v0);
    load_chunk(1, v1);
#pragma unroll
    for (int kt = 0; kt < 16; ++kt) {
      const uint4 x = ptx::ldg_nc_na_hint(rsrc + kt * 32, pol_first);
      wr[kt][0] = x.x;
      wr[kt][1] = x.y;
      wr[kt][2] = x.z;
      wr[kt][3] = x.w;
    }
#pragma unroll
    for (int p = 0; p < 8; p += 2) {
      store_chunk(p, v0);
      store_chunk(p + 1, v1);
      ptx::tmem_wait_st();
      if (p + 2 < 8) {
        load_chunk(p + 2, v0);
        load_chunk(p + 3, v1);
      }
    }
  }
  trace_stamp(a, a.gamma, 1);

  // step 0's u = W1[anchor]
  for (int b = warp; b < a.B; b += kResWarps) gather_u_row(a, tok_s[b], b, U, lane, 0);
  if (ra.S > 0 && threadIdx.x == 0) {
    if (!wait_mbar(&mbar[kMbarSmem], 0, t_entry, a.timeout_ns)) {
      abort_round(a.sync.hdr, round_s, kStatusTimeout);
      abort_s = 1;
    }
  }
  ptx::cp_async_wait_all();
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  trace_stamp(a, a.gamma, 2);

  const bool fast = fast_s != 0;
  const KeyPassMap kpm = key_pass_map(a.B, temp_s);
  const uint2 eseed = round_seed(a, round_s);             // this round's Philox key
  const int nslots = kpm.tpr >= 32 ? kpm.tpr / 32 : 1;   // group_best slots per request

  // ----------------------------------------------------------- the walk ---
  const uint32_t w2_addr = ptx::smem_u32(smem_w2);
  const uint32_t ring_addr = ptx::smem_u32(ring);
  const uint32_t blk0 =
      w2_addr + (uint32_t)warp * kSmemStripBytes + (lane >> 3) * 128 + (lane & 7) * 16;
  bool ok = abort_s == 0;
  int k = 0;
  for (; k < a.gamma && ok; ++k) {
    const uint64_t t_step = globaltimer_ns();
    trace_stamp(a, k, 0);

    // (0) streamed strips, groups of up to four: each strip's 16 k-tiles from
    // the ring, then the group's keys (greedy, no logits out) or logits
    if constexpr (STR) {
      if (fast && lane < a.B) warp_key[warp][lane] = 0u;
      __syncwarp();
      const uint32_t rw =
          ring_addr + (uint32_t)warp * kSmemStripBytes + (lane >> 3) * 128 + (lane & 7) * 16;
      for (int i0 = 0; i0 < nt2; i0 += kStreamGroup) {
        float accg[kStreamGroup][NT][4];
#pragma unroll
        for (int s = 0; s < kStreamGroup; ++s)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) accg[s][nt][e] = 0.0f;
#pragma unroll
        for (int ii = 0; ii < kStreamGroup; ++ii) {
          if (i0 + ii >= nt2) break;
          const int n = k * nt2 + i0 + ii;
          const int slot = n % nslot;
          if (!wait_mbar(&ring_bar[slot], (uint32_t)((n / nslot) & 1), t_step, a.timeout_ns) &&
              lane == 0) {
            abort_round(a.sync.hdr, round_s, kStatusTimeout);
            abort_s = 1;
          }
#pragma unroll
          for (int kt = 0; kt < 16; ++kt) {
            uint32_t f0, f1, f2, f3;
            ptx::ldmatrix_x4(rw + (uint32_t)slot * kRingSlotBytes + kt * 512, f0, f1, f2, f3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              uint32_t b0 = 0u, b1 = 0u;
              if (8 * nt + g < a.B) {
                b0 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + nt) * 128 + lane * 4);
                b1 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + 2 + nt) * 128 + lane * 4);
              }
              ptx::mma_16816(accg[ii][nt], f0, f1, f2, f3, b0, b1);
            }
          }
          __syncwarp();                    // every lane's reads of the slot are done
          if (lane == 0) {
            __threadfence_block();
            if (atomicSub(&ring_left[slot], 1) == 1) {   // the last warp: refill the slot
              ring_left[slot] = kMrWarps;
              __threadfence_block();
              if (n + nslot < ring_total) {
                ptx::fence_proxy_async_smem();
                ring_issue(n + nslot);
                atomicMax(ring_sent, n + nslot + 1);
              }
              atomicMax(ring_freed, n + 1);
            }
          }
        }
        const int st0 = 1 + kTmStrips + NS + i0;
        const int ng = nt2 - i0 < kStreamGroup ? nt2 - i0 : kStreamGroup;
        if (fast) {
          if constexpr (NT == 1) {
            if (a.B <= 2)
              fast_keys<kStreamGroup, 4, NT, true>(accg, 0, base_s, ra.R, a.B, nv, warp, lane,
                                                   &warp_key[warp][0], st0, ng);
            else if (a.B <= 4)
              fast_keys<kStreamGroup, 2, NT, true>(accg, 0, base_s, ra.R, a.B, nv, warp, lane,
                                                   &warp_key[warp][0], st0, ng);
            else
              fast_keys<kStreamGroup, 1, NT, true>(accg, 0, base_s, ra.R, a.B, nv, warp, lane,
                                                   &warp_key[warp][0], st0, ng);
          } else {
            fast_keys<kStreamGroup, 1, NT, true>(accg, 0, base_s, ra.R, a.B, nv, warp, lane,
                                                 &warp_key[warp][0], st0, ng);
            fast_keys<kStreamGroup, 1, NT, true>(accg, 1, base_s, ra.R, a.B, nv, warp, lane,
                                                 &warp_key[warp][0], st0, ng);
          }
        } else {
#pragma unroll
          for (int ii = 0; ii < kStreamGroup; ++ii)
            if (ii < ng) logits_strip<NT>(accg[ii], base_s, ra.R, a.B, strip_row0(st0 + ii, warp), lane);
        }
      }
    }

    // (1) projection: 16 k-tiles of up to 8 independent mma.sync chains (the
    // four tensor-memory strips, the register strip, the shared strips); the
    // tensor-memory fragments of k-tile pair p + 1 load while pair p computes
    float acc[NST][NT][4];
#pragma unroll
    for (int s = 0; s < NST; ++s)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[s][nt][e] = 0.0f;
    // the k-tile's A fragments of every strip against both n-tiles' B
    auto ktile = [&](int kt, const uint32_t* f) {     // f: the 4 strips' tensor-memory words
      uint32_t af[NS > 0 ? NS : 1][4];
#pragma unroll
      for (int j = 0; j < NS; ++j)
        ptx::ldmatrix_x4(blk0 + (uint32_t)(j * kResWarps) * kSmemStripBytes + kt * 512, af[j][0],
                         af[j][1], af[j][2], af[j][3]);
      uint32_t bf[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        bf[nt][0] = bf[nt][1] = 0u;
        if (8 * nt + g < a.B) {            // this lane's B-fragment column is a request
          bf[nt][0] = *reinterpret_cast<const uint32_t*>(U + (4 * kt + nt) * 128 + lane * 4);
          bf[nt][1] = *reinterpret_cast<const uint32_t*>(U + (4 * kt + 2 + nt) * 128 + lane * 4);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int s = 0; s < kTmStrips; ++s)
          ptx::mma_16816(acc[s][nt], f[4 * s], f[4 * s + 1], f[4 * s + 2], f[4 * s + 3],
                         bf[nt][0], bf[nt][1]);
        ptx::mma_16816(acc[kTmStrips][nt], wr[kt][0], wr[kt][1], wr[kt][2], wr[kt][3],
                       bf[nt][0], bf[nt][1]);
#pragma unroll
        for (int j = 0; j < NS; ++j)
          ptx::mma_16816(acc[1 + kTmStrips + j][nt], af[j][0], af[j][1], af[j][2], af[j][3],
                         bf[nt][0], bf[nt][1]);
      }
    };
    if constexpr (NT == 1) {
      // one 32-column load per k-tile pair, one pair ahead
      uint32_t fr[2][32];
      ptx::tmem_ld32(tm_addr, fr[0]);
      ptx::tmem_wait_ld32(fr[0]);
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (p + 1 < 8) ptx::tmem_ld32(tm_addr + 32 * (p + 1), fr[(p + 1) & 1]);
        ktile(2 * p, &fr[p & 1][0]);
        ktile(2 * p + 1, &fr[p & 1][16]);
        if (p + 1 < 8) ptx::tmem_wait_ld32(fr[(p + 1) & 1]);
      }
    } else {
      // twice the accumulators: one 16-column load per k-tile, one ahead
      uint32_t fr[2][16];
      ptx::tmem_ld<16>(tm_addr, fr[0]);
      ptx::tmem_wait_ld16(fr[0]);
#pragma unroll
      for (int kt = 0; kt < 16; ++kt) {
        if (kt + 1 < 16) ptx::tmem_ld<16>(tm_addr + 16 * (kt + 1), fr[(kt + 1) & 1]);
        ktile(kt, fr[kt & 1]);
        if (kt + 1 < 16) ptx::tmem_wait_ld16(fr[(kt + 1) & 1]);
      }
    }
    trace_stamp(a, k, 1);

    // (2) epilogue
    if (fast) {
      // greedy, no logits out: keys straight from the accumulators
      if constexpr (NT == 1) {
        if (a.B <= 2)
          fast_keys<NST, 4, NT, STR>(acc, 0, base_s, ra.R, a.B, nv, warp, lane, &warp_key[warp][0]);
        else if (a.B <= 4)
          fast_keys<NST, 2, NT, STR>(acc, 0, base_s, ra.R, a.B, nv, warp, lane, &warp_key[warp][0]);
        else
          fast_keys<NST, 1, NT, STR>(acc, 0, base_s, ra.R, a.B, nv, warp, lane, &warp_key[warp][0]);
      } else {
        fast_keys<NST, 1, NT, STR>(acc, 0, base_s, ra.R, a.B, nv, warp, lane, &warp_key[warp][0]);
        fast_keys<NST, 1, NT, STR>(acc, 1, base_s, ra.R, a.B, nv, warp, lane, &warp_key[warp][0]);
      }
      trace_stamp(a, k, 2);
      trace_stamp(a, k, 3);
      __syncthreads();
    } else {
      // logits into the shared base buffer (in place), then the key pass
#pragma unroll
      for (int s = 0; s < NST; ++s)           // (a padding strip's rows lie past R)
        if (strip_row0(s, warp) < ra.R)
          logits_strip<NT>(acc[s], base_s, ra.R, a.B, strip_row0(s, warp), lane);
      trace_stamp(a, k, 2);
      __syncthreads();
      key_pass<(NT > 1)>(a, base_s, ra.R, nv, row0, k, kpm, eseed, group_best);
      trace_stamp(a, k, 3);
      __syncthreads();
    }
    trace_stamp(a, k, 4);

    // (3) the rendezvous.  Post: this CTA's best key of request b goes into
    // its own tagged slot, one relaxed store (the tag validates the word, so
    // no fence orders it and no atomic contends for a line).  Then every warp
    // starts the next step's base rows, and warp b polls request b's slots of
    // all CTAs until each carries this round's tag, takes the maximum and
    // puts the winner's W1 row into U.  Up to 8 requests, the row of the best
    // key seen so far is loaded while the last keys arrive, so that when the
    // winner posted early its row is already on the way.
    //
    // On GB300 another SM's poll sees a store 420-440 ns after it issues (for
    // every store and load form tried), against ~150 ns for a load's round
    // trip; so each poll keeps all of its slot loads in flight at once (a
    // fixed trip count over at most kMrMaxCtas slots), and the maximum of a
    // poll is two redux.sync (two per half-warp above 8 requests).
    const uint32_t parity = round_s & 1u;
    const unsigned long long tag = slot_tag(round_s);
    if (warp == 0 && lane < a.B) {
      unsigned long long mine = 0ull;
      if (fast) {
        uint32_t m = 0u;
#pragma unroll
        for (int w = 0; w < kMrWarps; ++w) m = max_u32(m, warp_key[w][lane]);
        if (m != 0u) {
          const uint32_t v = (uint32_t)(row0 + (0xFFFFu - (m & 0xFFFFu)));
          mine = ((unsigned long long)(m >> 16) << 32) | (unsigned long long)(0xFFFFFFFFu - v);
        }
      } else {
        for (int sl = 0; sl < nslots; ++sl) mine = key_max(mine, group_best[lane][sl]);
      }
      if (cta != a.skip_cta) {
        st_relaxed_gpu_u64(a.sync.slot_at(parity, k, lane) + cta, tag | key50(mine));
        red_relaxed_gpu_add(a.sync.count_at(parity, k) + lane, 1u);   // a hint, see below
      }
      if (mine != 0ull) {                          // the candidate's W1 row, into L2
        const uint16_t* row = a.W1 + (size_t)(0xFFFFFFFFu - (uint32_t)mine) * kRank;
#pragma unroll
        for (int i = 0; i < 4; ++i) ptx::prefetch_l2(row + 64 * i);
      }
    }
    trace_stamp(a, k, 5);
    prefetch_base(ra, k + 1, row0, nv, base_s);
    if (NT == 1 && warp < a.B) {     // warp w takes request w
      const unsigned long long* s = a.sync.slot_at(parity, k, warp);
      unsigned long long best = 0ull;
      int good = 1;
      uint32_t spins = 0;
      // lane 0 first waits until three quarters of the CTAs have counted in
      // (one word: far less polling traffic than every warp reading every
      // slot); the count carries no ordering, the slots' tags decide.  Then
      // the warp reads all slots until every tag is this round's: a slot not
      // yet written of this parity holds 0, so the maximum so far is a lower
      // bound of the winner, and its W1 row is loaded into rowv whenever it
      // changes (the last load is the winner's)
      if (lane == 0) {
        const uint32_t* cp = a.sync.count_at(parity, k) + warp;
        const uint32_t early = (uint32_t)(n_cta - (n_cta >> 2));
        while (ld_relaxed_gpu_u32(cp) < early) {
          if ((++spins & 63u) == 0u &&
              (round_aborted(a.sync.hdr, round_s) ||
               (int64_t)(globaltimer_ns() - t_step) > a.timeout_ns))
            break;                     // the slot loop below reports it
        }
      }
      __syncwarp();
      spins = 0;
      unsigned long long cand = 0ull;                  // the key whose row rowv holds
      uint4 rowv = make_uint4(0u, 0u, 0u, 0u);
      while (true) {
        bool have = true;
        best = 0ull;
        {
          // every slot load of a poll in flight together (a fixed trip count;
          // a loop bounded by the CTA count issued them one round trip apart)
          constexpr int nld = kMrMaxCtas / 64;
          unsigned long long xx[nld][2];
#pragma unroll
          for (int it = 0; it < nld; ++it) {
            const int j = 2 * lane + 64 * it;
            if (j < n_cta) {
              ld_relaxed_gpu_v2u64(s + j, xx[it][0], xx[it][1]);
            } else {
              xx[it][0] = tag;
              xx[it][1] = tag;
            }
          }
#pragma unroll
          for (int it = 0; it < nld; ++it) {
            const int j = 2 * lane + 64 * it;
            if (j + 1 >= n_cta) xx[it][1] = tag;       // the padding word after an odd count
            have = have && (xx[it][0] & ~kKey50Mask) == tag && (xx[it][1] & ~kKey50Mask) == tag;
            const unsigned long long x0 = xx[it][0] & kKey50Mask, x1 = xx[it][1] & kKey50Mask;
            best = x0 > best ? x0 : best;
            best = x1 > best ? x1 : best;
          }
        }
        const bool all = __all_sync(0xFFFFFFFFu, have);
        {                                            // the 50-bit maximum as two 32-bit ones
          const uint32_t hi = (uint32_t)(best >> 32), mh = ptx::redux_max_u32(hi);
          const uint32_t ml = ptx::redux_max_u32(hi == mh ? (uint32_t)best : 0u);
          best = ((unsigned long long)mh << 32) | ml;
        }
        if (best != cand && best != 0ull && k + 1 < a.gamma) {
          const int32_t t = key50_token(best);
          if (t >= 0 && (int64_t)t < a.V) {
            cand = best;
            rowv = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)t * kRank) + lane);
          }
        }
        if (all) break;
        if ((++spins & 15u) == 0u) {
          int stop = 0;
          if (lane == 0) {
            if (round_aborted(a.sync.hdr, round_s)) {
              stop = 1;
            } else if ((int64_t)(globaltimer_ns() - t_step) > a.timeout_ns) {
              abort_round(a.sync.hdr, round_s, kStatusTimeout);
              stop = 1;
            }
          }
          if (__shfl_sync(0xFFFFFFFFu, stop, 0)) {
            good = 0;
            break;
          }
        }
      }
      if (good) {
        if (warp == 0) trace_stamp(a, k, 6);
        const int32_t tok = key50_token(best);
        if (tok < 0 || (int64_t)tok >= a.V) {      // cannot happen: every CTA posts a real row
          if (lane == 0) {
            abort_round(a.sync.hdr, round_s, kStatusInternal);
            abort_s = 1;
          }
        } else {
          if (lane == 0) {
            tok_s[warp] = tok;
            if (cta == 0) a.out_tokens[(size_t)warp * a.gamma + k] = tok;
          }
          if (k + 1 < a.gamma)       // rowv holds W1[tok]: cand == best here
            *reinterpret_cast<uint4*>(U + (lane * 2 + (warp >> 3)) * 128 + (warp & 7) * 16) = rowv;
        }
      } else if (lane == 0) {
        abort_s = 1;
      }
    }
    // above 8 requests each half-warp of warp w takes one, requests w and
    // w + 8 side by side
    constexpr int halves = 2;                            // B > 8 exactly when NT = 2
    constexpr int span = 32 / halves;                    // lanes per request
    const int li = lane % span;                          // lane within the request's lanes
    const int rq = warp + kResWarps * (lane / span);
    if (NT == 2 && warp < a.B) {
      const bool mine = rq < a.B;
      const unsigned long long* s = a.sync.slot_at(parity, k, mine ? rq : warp);
      unsigned long long best = 0ull;
      int good = 1;
      uint32_t spins = 0;
      // as above: the first lane of a request waits until three quarters of
      // the CTAs have counted in, then the request's lanes read the slots
      // until every tag is this round's, loading the row of the best key so
      // far whenever it changes
      if (li == 0 && mine) {
        const uint32_t* cp = a.sync.count_at(parity, k) + rq;
        const uint32_t early = (uint32_t)(n_cta - (n_cta >> 2));
        while (ld_relaxed_gpu_u32(cp) < early) {
          if ((++spins & 63u) == 0u &&
              (round_aborted(a.sync.hdr, round_s) ||
               (int64_t)(globaltimer_ns() - t_step) > a.timeout_ns))
            break;                     // the slot loop below reports it
        }
      }
      __syncwarp();
      spins = 0;
      constexpr int nchunk = 32 / span;                  // 16-byte chunks of the row per lane
      unsigned long long cand = 0ull;
      uint4 rowv[nchunk];
#pragma unroll
      for (int i = 0; i < nchunk; ++i) rowv[i] = make_uint4(0u, 0u, 0u, 0u);
      while (true) {
        bool have = true;
        best = 0ull;
        if (mine) {
          constexpr int nld = kMrMaxCtas / (2 * span);
          unsigned long long xx[nld][2];
#pragma unroll
          for (int it = 0; it < nld; ++it) {
            const int j = 2 * li + 2 * span * it;
            if (j < n_cta) {
              ld_relaxed_gpu_v2u64(s + j, xx[it][0], xx[it][1]);
            } else {
              xx[it][0] = tag;
              xx[it][1] = tag;
            }
          }
#pragma unroll
          for (int it = 0; it < nld; ++it) {
            const int j = 2 * li + 2 * span * it;
            if (j + 1 >= n_cta) xx[it][1] = tag;
            have = have && (xx[it][0] & ~kKey50Mask) == tag && (xx[it][1] & ~kKey50Mask) == tag;
            const unsigned long long x0 = xx[it][0] & kKey50Mask, x1 = xx[it][1] & kKey50Mask;
            best = x0 > best ? x0 : best;
            best = x1 > best ? x1 : best;
          }
        }
        const bool all = __all_sync(0xFFFFFFFFu, have);
        {                                                // each half-warp's 50-bit maximum
          const bool upper = lane >= 16;
          const uint32_t h = (uint32_t)(best >> 32);
          const uint32_t h0 = ptx::redux_max_u32(upper ? 0u : h);
          const uint32_t h1 = ptx::redux_max_u32(upper ? h : 0u);
          const uint32_t mh = upper ? h1 : h0;
          const uint32_t l = h == mh ? (uint32_t)best : 0u;
          const uint32_t l0 = ptx::redux_max_u32(upper ? 0u : l);
          const uint32_t l1 = ptx::redux_max_u32(upper ? l : 0u);
          best = ((unsigned long long)mh << 32) | (upper ? l1 : l0);
        }
        if (mine && best != cand && best != 0ull && k + 1 < a.gamma) {
          const int32_t t = key50_token(best);
          if (t >= 0 && (int64_t)t < a.V) {
            cand = best;
#pragma unroll
            for (int i = 0; i < nchunk; ++i)
              rowv[i] = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)t * kRank) + li + span * i);
          }
        }
        if (all) break;
        if ((++spins & 15u) == 0u) {
          int stop = 0;
          if (lane == 0) {
            if (round_aborted(a.sync.hdr, round_s)) {
              stop = 1;
            } else if ((int64_t)(globaltimer_ns() - t_step) > a.timeout_ns) {
              abort_round(a.sync.hdr, round_s, kStatusTimeout);
              stop = 1;
            }
          }
          if (__shfl_sync(0xFFFFFFFFu, stop, 0)) {
            good = 0;
            break;
          }
        }
      }
      if (good) {
        if (rq == 0) trace_stamp(a, k, 6);
        const int32_t tok = key50_token(best);
        if (mine && (tok < 0 || (int64_t)tok >= a.V)) {   // cannot happen: real rows only
          if (li == 0) {
            abort_round(a.sync.hdr, round_s, kStatusInternal);
            abort_s = 1;
          }
        } else if (mine) {
          if (li == 0) {
            tok_s[rq] = tok;
            if (cta == 0) a.out_tokens[(size_t)rq * a.gamma + k] = tok;
          }
          if (k + 1 < a.gamma)                 // rowv holds W1[tok]'s chunks li + span i
#pragma unroll
            for (int i = 0; i < nchunk; ++i) {
              const int c = li + span * i;
              *reinterpret_cast<uint4*>(U + (c * 2 + (rq >> 3)) * 128 + (rq & 7) * 16) = rowv[i];
            }
        }
      } else if (lane == 0) {
        abort_s = 1;
      }
    }
    ptx::cp_async_wait_all();
    __syncthreads();
    trace_stamp(a, k, 7);
    ok = abort_s == 0;
  }

  // -------------------------------------------------------------- exit ----
  ptx::tc_fence_before();
  __syncthreads();
  // a walk that stopped early may leave ring copies in flight: let them land
  // before the CTA's shared memory goes away
  if (STR && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (int n = *ring_freed; n < *ring_sent; ++n)
      (void)wait_mbar(&ring_bar[n % nslot], (uint32_t)((n / nslot) & 1), t0, a.timeout_ns);
  }
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
  if (cta == 0) {
    if (!ok)
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    if (threadIdx.x == 0) atomicAdd(&a.sync.hdr->round, 1u);
  }
  trace_stamp(a, a.gamma, 4);          // the CTA's last
}

// Position (local row, K word pair) of word i of a CTA's block of the repacked
// W2 (see the tier layouts above); the repack and its inverse share it.
__device__ __forceinline__ void mr_word_pos(int64_t i, int* rl, int* kp) {
  if (i < kTmWords) {           // [warp][p][m][lane][4]
    const int j4 = (int)(i & 3), l = (int)((i >> 2) & 31), m = (int)((i >> 7) & 7);
    const int p = (int)((i >> 10) & 7), w = (int)(i >> 13);
    const int ii = 4 * m + j4;                 // word of lane l's 32-column chunk p
    const int e = ii >> 4, s = (ii >> 2) & 3, j = ii & 3;
    const int kt = 2 * p + e;
    *rl = 16 * (kTmStrips * w + s) + (l >> 2) + 8 * (j & 1);
    *kp = kt * 8 + (l & 3) + 4 * (j >> 1);
  } else if (i < kTmWords + kMrRfWords) {    // [warp][kt][lane][4]
    const int64_t x = i - kTmWords;
    const int j = (int)(x & 3), l = (int)((x >> 2) & 31), kt = (int)((x >> 7) & 15);
    const int w = (int)(x >> 11);
    *rl = kTmRows + 16 * w + (l >> 2) + 8 * (j & 1);
    *kp = kt * 8 + (l & 3) + 4 * (j >> 1);
  } else {                                   // [strip][kt][matrix][row][4] (ldmatrix)
    const int64_t x = i - kTmWords - kMrRfWords;
    const int p = (int)(x & 3), ii = (int)((x >> 2) & 7), m = (int)((x >> 5) & 3);
    const int kt = (int)((x >> 7) & 15), s2 = (int)(x >> 11);
    *rl = kMrFixedRows + 16 * s2 + 8 * (m & 1) + ii;
    *kp = kt * 8 + 4 * (m >> 1) + p;
  }
}

// Repack row-major W2 [V, 256] (32-bit words of two K elements) into the
// per-CTA tiered layout (rows past V are zero), or, with `inverse`, write the
// rows held in the layout back to row-major form.
__global__ void repack_mma_kernel(uint32_t* __restrict__ rowmajor, uint32_t* __restrict__ packed,
                                  int64_t V, int R, int64_t words_per_cta, int n_cta,
                                  int inverse) {
  const int64_t total = words_per_cta * n_cta;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t cta = i / words_per_cta;
    int rl, kp;
    mr_word_pos(i - cta * words_per_cta, &rl, &kp);
    const int64_t row = cta * (int64_t)R + rl;
    if (inverse) {
      if (row < V) rowmajor[row * (kRank / 2) + kp] = packed[i];
    } else {
      packed[i] = row < V ? rowmajor[row * (kRank / 2) + kp] : 0u;
    }
  }
}

}  // namespace

int mma_resident_fixed_rows() { return kMrFixedRows; }

int mma_resident_max_rows() { return kMrMaxRows; }

int mma_resident_max_batch() { return kMrMaxB; }

int mma_resident_max_ctas() { return kMrMaxCtas; }

int64_t mma_resident_words_per_cta(int S) {
  return (int64_t)kTmWords + kMrRfWords + (int64_t)S * (kSmemStripBytes / 4);
}

size_t mma_resident_smem_bytes(int S, int max_B, int R, int nslot) {
  return (size_t)S * kSmemStripBytes +
         (nslot > 0 ? (size_t)nslot * kRingSlotBytes + kRingCtlBytes : 0) + 16 * 512 +
         (((size_t)max_B * R * 2 + 15) & ~(size_t)15);
}

const void* mma_resident_kernel(int S, int NT, bool streamed) {
  const int NS = (S + kMrWarps - 1) / kMrWarps;
  if (streamed) {
    if (NT == 1) {
      switch (NS) {
        case 0: return reinterpret_cast<const void*>(&walk_mma_kernel<0, 1, true>);
        case 1: return reinterpret_cast<const void*>(&walk_mma_kernel<1, 1, true>);
        case 2: return reinterpret_cast<const void*>(&walk_mma_kernel<2, 1, true>);
      }
    } else if (NT == 2) {
      switch (NS) {
        case 0: return reinterpret_cast<const void*>(&walk_mma_kernel<0, 2, true>);
        case 1: return reinterpret_cast<const void*>(&walk_mma_kernel<1, 2, true>);
        case 2: return reinterpret_cast<const void*>(&walk_mma_kernel<2, 2, true>);
      }
    }
    return nullptr;
  }
  if (NT == 1) {
    switch (NS) {
      case 0: return reinterpret_cast<const void*>(&walk_mma_kernel<0, 1, false>);
      case 1: return reinterpret_cast<const void*>(&walk_mma_kernel<1, 1, false>);
      case 2: return reinterpret_cast<const void*>(&walk_mma_kernel<2, 1, false>);
      case 3: return reinterpret_cast<const void*>(&walk_mma_kernel<3, 1, false>);
    }
  } else if (NT == 2) {
    switch (NS) {
      case 0: return reinterpret_cast<const void*>(&walk_mma_kernel<0, 2, false>);
      case 1: return reinterpret_cast<const void*>(&walk_mma_kernel<1, 2, false>);
      case 2: return reinterpret_cast<const void*>(&walk_mma_kernel<2, 2, false>);
      case 3: return reinterpret_cast<const void*>(&walk_mma_kernel<3, 2, false>);
    }
  }
  return nullptr;
}

cudaError_t mma_resident_repack(void* rowmajor, void* packed, int64_t V, int R, int S, int n_cta,
                                bool inverse, cudaStream_t stream) {
  const int64_t wpc = mma_resident_words_per_cta(S);
  const int64_t total = wpc * n_cta;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  repack_mma_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint32_t*>(rowmajor),
                                               static_cast<uint32_t*>(packed), V, R, wpc, n_cta,
                                               inverse ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace dspark
