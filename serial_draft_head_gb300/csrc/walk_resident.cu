// walk_resident.cu -- the persistent walk with W2 held on chip for the whole
// round: "Keeping the Draft Walk on Chip: One Launch for DSpark's Markov
// Head", sections "The idea: make the walk resident" (one CTA per SM, one
// launch per round, each CTA loads its slice of rows once and runs all gamma
// steps) and "B200: the bf16 table fits on chip" (the table split over
// tensor memory, shared memory and registers; tcgen05 reads the tensor-memory
// part, mma.sync the rest; request n is column n of the MMA's N operand).
//
// Per CTA (256 threads, 8 warps) the R rows of its shard are placed as
//   rows [0, 384)             3 tiles of 128 rows in tensor memory, read by
//                             tcgen05.mma (A from TMEM, B = U from shared
//                             memory, D = two 128 x 16 fp32 partial sums per
//                             tile, one per K half, in TMEM);
//   rows [384, 384 + 128 RS)  registers: each warp holds RS 16-row strips as
//                             mma.sync A fragments;
//   rows [384 + 128 RS, R)    shared memory, 16-row strips read by ldmatrix
//                             and mma.sync.
//   rows [.., R)              when the shard does not fit on chip ("V = 248,320:
//                             62% on chip, the rest streamed"): ST strips in
//                             the shared-strip layout, streamed every step
//                             through a ring of two or three 64 KB slots (8
//                             strips each) by bulk copies; the ring keeps
//                             refilling across steps since W2 does not depend
//                             on the token.  Warp w reads strip w of a slot.
// U (the gathered W1 rows, one per request) sits in shared memory in the
// no-swizzle K-major core-matrix layout that both the tcgen05 descriptor and
// the mma.sync B fragments read.
//
// Cross-CTA selection follows the blog post's rendezvous: per step and
// request an atomic max of the 64-bit {logit order bits, inverted id} key,
// released by an atomic arrival count that one thread per CTA polls.  (A
// gather variant in which every CTA reads every CTA's slot measured 2.6 us
// per step at 151 CTAs on GB300 against 1.5 us for the atomics: 151 readers
// of the same few L2 lines contend.)
#include "resident_pass.cuh"
#include "tc_ptx.cuh"
#include "walk_common.cuh"
#include "walk_kernels.h"

namespace dspark {

namespace {

constexpr int kTmemTiles = 3;
constexpr int kTmemCols = 512;
constexpr int kTmemRows = kTmemTiles * 128;    // rows held in tensor memory
constexpr int kDCol0 = kTmemTiles * 128;       // first accumulator column
constexpr int kIssuers = 2 * kTmemTiles;       // one per (tile, K half)
constexpr int kMbarTma = kIssuers;             // mbarrier of the shared-tier bulk copy
constexpr int kNMma = 16;                      // tcgen05 N (requests per MMA)
constexpr int kTmemWords = kTmemTiles * 128 * 128;
constexpr int kRfStripWords = kResWarps * 16 * 32 * 4;  // one strip per warp, all warps
constexpr int kChunkStrips = 8;                // streamed strips per ring slot
constexpr int kChunkBytes = kChunkStrips * kSmemStripBytes;
constexpr int kMaxRingSlots = 3;
constexpr int kMbarRing = kMbarTma + 1;        // first of the ring slots' mbarriers
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, kNMma);
static_assert(kResThreads == kRank, "one thread per state element");


// CELL: the instantiation that also runs the recurrent heads and writes the
// state output (the Markov-only one carries none of that code).
// A recurrent head's next state for request b, lane l's elements 8l .. 8l + 7
// (p from L2, the winner's W1 row, the current state in U, updated in place).
__device__ __forceinline__ void cell_update_row(const WalkArgs& a, uint8_t* U, int k, int b,
                                                int32_t tok, int lane) {
  const float4* pp =
      reinterpret_cast<const float4*>(a.cell_p + ((size_t)k * 16 + b) * kCellP) + 2 * lane;
  const float4 p0 = __ldcg(pp), p1 = __ldcg(pp + 1);
  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok * kRank) + lane);
  uint4* hp = reinterpret_cast<uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16);
  const uint4 hv = *hp;
  const float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
  uint32_t ow[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t lo = cell_element(a.cell, p[2 * e], bf16_bits_to_float(xw[e] & 0xFFFFu),
                                     bf16_bits_to_float(hw[e] & 0xFFFFu));
    const uint32_t hi = cell_element(a.cell, p[2 * e + 1], bf16_bits_to_float(xw[e] >> 16),
                                     bf16_bits_to_float(hw[e] >> 16));
    ow[e] = lo | (hi << 16);
  }
  *hp = make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// The GRU's next state for request b, lane l's elements 8l .. 8l + 7: the
// three recurrent products and the token's three table rows, one 16-byte
// chunk (two for the fp32 products) of each per lane.
__device__ __forceinline__ void gru_update_row(const WalkArgs& a, uint8_t* U, int k, int b,
                                               int32_t tok, int lane) {
  const float4* pp =
      reinterpret_cast<const float4*>(a.cell_p + ((size_t)k * 16 + b) * kCellP) + 2 * lane;
  const uint4* X = reinterpret_cast<const uint4*>(a.cell_X);
  float4 pv[6];
#pragma unroll
  for (int g = 0; g < 3; ++g) {
    pv[2 * g] = __ldcg(pp + g * (kRank / 4));
    pv[2 * g + 1] = __ldcg(pp + g * (kRank / 4) + 1);
  }
  uint4 xv[3];
#pragma unroll
  for (int g = 0; g < 3; ++g) xv[g] = __ldg(X + ((size_t)g * a.V + tok) * 32 + lane);
  uint4* hp = reinterpret_cast<uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16);
  const uint4 hv = *hp;
  const float* pf = reinterpret_cast<const float*>(pv);          // [gate][8]
  const uint32_t* xw = reinterpret_cast<const uint32_t*>(xv);   // [gate][4]
  const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
  uint32_t ow[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint32_t half[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int j = 2 * e + t;
      const int sh = 16 * t;
      half[t] = gru_element(pf[j], pf[8 + j], pf[16 + j],
                            bf16_bits_to_float((xw[e] >> sh) & 0xFFFFu),
                            bf16_bits_to_float((xw[4 + e] >> sh) & 0xFFFFu),
                            bf16_bits_to_float((xw[8 + e] >> sh) & 0xFFFFu),
                            bf16_bits_to_float((hw[e] >> sh) & 0xFFFFu));
    }
    ow[e] = half[0] | (half[1] << 16);
  }
  *hp = make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

template <int RS, int NT, int SMAX, bool CELL>
__global__ void __launch_bounds__(kResThreads, 1) walk_resident_kernel(const ResidentArgs ra) {
  constexpr int NCOL = 8 * NT;
  const WalkArgs& a = ra.w;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* smem_w2 = smem;
  uint8_t* ring = smem + (size_t)ra.S * kSmemStripBytes;
  const int nslot = ra.ST > 0 ? ra.nslot : 0;    // ring slots of kChunkBytes
  uint8_t* U = ring + (size_t)nslot * kChunkBytes;
  uint16_t* base_s = reinterpret_cast<uint16_t*>(U + 16 * 512);
  __shared__ __align__(8) uint64_t mbar[kMbarRing + kMaxRingSlots];
  __shared__ int slot_done[kMaxRingSlots];
  __shared__ int ring_issued, ring_consumed;
  __shared__ unsigned long long group_best[16][kResWarps];
  __shared__ float temp_s[16];
  __shared__ int32_t tok_s[16];
  __shared__ uint32_t tmem_base_s;
  __shared__ int flag_s;
  __shared__ int abort_s;
  __shared__ uint32_t round_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int cta = blockIdx.x;
  const int n_cta = gridDim.x;
  const int64_t row0 = (int64_t)cta * ra.R;
  const int nv = (int)((a.V - row0) < ra.R ? (a.V - row0) : ra.R);  // valid rows (>= 1)
  const uint32_t* gw = ra.W2p + (size_t)cta * (size_t)ra.words_per_cta;

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
    for (int i = 0; i < kMbarRing + kMaxRingSlots; ++i) ptx::mbar_init(&mbar[i], 1);
    for (int i = 0; i < kMaxRingSlots; ++i) slot_done[i] = 0;
    ring_issued = ring_consumed = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&tmem_base_s, kTmemCols);
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

  // the other parity's keys and counts start empty for the next round
  if (cta == 0) clear_other_parity(a.sync, round_s & 1u);

  // shared-memory tier: bulk copies straight to its final place
  const uint64_t t_entry = globaltimer_ns();
  if (threadIdx.x == 0 && ra.S > 0) {
    const uint32_t bytes = (uint32_t)ra.S * kSmemStripBytes;
    ptx::mbar_expect_tx(&mbar[kMbarTma], bytes);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(gw + kTmemWords + RS * kRfStripWords);
    for (uint32_t off = 0; off < bytes; off += 32768u) {
      const uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
      ptx::bulk_g2s(smem_w2 + off, src + off, n, &mbar[kMbarTma]);
    }
  }

  // streamed tier: the first two chunks of step 0 into the ring
  const uint8_t* gstream = reinterpret_cast<const uint8_t*>(gw + kTmemWords + RS * kRfStripWords) +
                           (size_t)ra.S * kSmemStripBytes;
  const int n_chunks = (ra.ST + kChunkStrips - 1) / kChunkStrips;   // per step
  auto issue_chunk = [&](int gi) {    // chunk gi of the round (step gi / n_chunks), slot gi % nslot
    const int c = gi % n_chunks;
    const int ns = ra.ST - c * kChunkStrips < kChunkStrips ? ra.ST - c * kChunkStrips : kChunkStrips;
    const uint32_t bytes = (uint32_t)ns * kSmemStripBytes;
    uint64_t* bar = &mbar[kMbarRing + gi % nslot];
    ptx::mbar_expect_tx(bar, bytes);
    // re-read every step: evict-last, so that it stays in L2 across the steps
    ptx::bulk_g2s_hint(ring + (size_t)(gi % nslot) * kChunkBytes,
                       gstream + (size_t)c * kChunkBytes, bytes, bar, ptx::policy_evict_last());
  };
  if (threadIdx.x == 0 && ra.ST > 0) {
    const int pre = a.gamma * n_chunks < nslot ? a.gamma * n_chunks : nslot;
    for (int gi = 0; gi < pre; ++gi) issue_chunk(gi);
    ring_issued = pre;
  }

  // step 0's base rows: asynchronous copies, in flight during the loads below
  prefetch_base(ra, 0, row0, nv, base_s);

  // tensor-memory tier: global -> registers -> tcgen05.st (warp w writes lane
  // quarter w % 4, column half w / 4 of every tile).  Tiles 0 and 1 are in
  // flight together; tile 2 shares its round trip with the register tier.
  const int tq = warp & 3, th = warp >> 2;
  const uint4* tsrc = reinterpret_cast<const uint4*>(gw);
  auto load_tile = [&](int t, uint32_t (&v)[4][16]) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 x = __ldg(tsrc + ((((t * 2 + th) * 16 + c) * 4 + tq) * 32 + lane));
      v[c >> 2][(c & 3) * 4 + 0] = x.x;
      v[c >> 2][(c & 3) * 4 + 1] = x.y;
      v[c >> 2][(c & 3) * 4 + 2] = x.z;
      v[c >> 2][(c & 3) * 4 + 3] = x.w;
    }
  };
  auto store_tile = [&](int t, uint32_t (&v)[4][16]) {
#pragma unroll
    for (int part = 0; part < 4; ++part)
      ptx::tmem_st16(tmem + ((uint32_t)(32 * tq) << 16) + t * 128 + 64 * th + part * 16, v[part]);
  };
  {
    uint32_t v0[4][16], v1[4][16];
    load_tile(0, v0);
    load_tile(1, v1);
    store_tile(0, v0);
    store_tile(1, v1);
  }
  uint32_t wr[RS][16][4];              // register tier: this warp's RS strips as A fragments
  {
    uint32_t v2[4][16];
    load_tile(2, v2);
    const uint4* src = reinterpret_cast<const uint4*>(gw + kTmemWords) +
                       (size_t)(warp * RS) * 16 * 32 + lane;
#pragma unroll
    for (int s = 0; s < RS; ++s)
#pragma unroll
      for (int kt = 0; kt < 16; ++kt) {
        const uint4 x = __ldg(src + (s * 16 + kt) * 32);
        wr[s][kt][0] = x.x;
        wr[s][kt][1] = x.y;
        wr[s][kt][2] = x.z;
        wr[s][kt][3] = x.w;
      }
    store_tile(2, v2);
  }
  ptx::tmem_wait_st();
  trace_stamp(a, a.gamma, 1);

  // step 0's u = W1[anchor]
  for (int b = warp; b < a.B; b += kResWarps)
    gather_u_row(a, tok_s[b], b, U, lane, CELL ? a.cell : 0);
  if (ra.S > 0 && threadIdx.x == 0) {
    if (!wait_mbar(&mbar[kMbarTma], 0, t_entry, a.timeout_ns)) {
      abort_round(a.sync.hdr, round_s, kStatusTimeout);
      abort_s = 1;
    }
  }
  ptx::cp_async_wait_all();
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  trace_stamp(a, a.gamma, 2);

  // a recurrent head's row of M for this warp (see publish_cell_rows)
  uint4 mreg = make_uint4(0u, 0u, 0u, 0u);
  if (CELL && a.cell != 0 && a.cell_q <= kResWarps) {
    const int row = cta * a.cell_q + warp % a.cell_q;
    if (row < (a.cell == 3 ? kCellP : kRank))
      mreg = __ldg(reinterpret_cast<const uint4*>(a.cell_M + (size_t)row * kRank) + lane);
  }
  const KeyPassMap kpm = key_pass_map(a.B, temp_s);
  const uint2 eseed = round_seed(a, round_s);             // this round's Philox key
  const int nslots = kpm.tpr >= 32 ? kpm.tpr / 32 : 1;   // group_best slots per request

  // ----------------------------------------------------------- the walk ---
  const uint32_t u_addr = ptx::smem_u32(U);
  const uint32_t w2_addr = ptx::smem_u32(smem_w2);
  bool ok = abort_s == 0;
  int k = 0;
  for (; k < a.gamma && ok; ++k) {
    ptx::tc_fence_after();
    const uint64_t t_step = globaltimer_ns();
    trace_stamp(a, k, 0);
    if (CELL && a.out_state != nullptr && cta == 0)   // this step's latent (the state)
      for (int b = 0; b < a.B; ++b)
        a.out_state[((size_t)b * a.gamma + k) * kRank + threadIdx.x] = *u_elem(U, threadIdx.x, b);

    // (1) tensor-memory tiles: a single thread issues one tcgen05.mma per ~45
    // cycles, so six warps each issue one (tile, K half): 8 MMAs into their
    // own 16-column partial accumulator, committed to their own mbarrier
    if (lane == 0 && warp < kIssuers) {
      const int t = warp >> 1, h = warp & 1;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int kt = 8 * h + kk;
        const uint64_t bdesc = ptx::smem_desc_noswizzle(u_addr + kt * 512, 256, 128);
        ptx::tc_mma_tmem_a(tmem + kDCol0 + 16 * warp, tmem + t * 128 + kt * 8, bdesc, kIdesc,
                           kk > 0 ? 1u : 0u);
      }
      ptx::tc_commit(&mbar[warp]);
    }
    __syncwarp();

    // streamed strips: chunk after chunk through the ring; the last warp done
    // with a slot refills it with the chunk nslot ahead (the next step's first
    // chunks load while this step finishes).  The chunks already in the ring
    // go first, so that their refills overlap the register/shared strips.
    const uint32_t ring_addr = ptx::smem_u32(ring);
    auto consume_chunk = [&](int c) -> bool {
      const int gc = k * n_chunks + c, slot = gc % nslot;
      if (!wait_mbar(&mbar[kMbarRing + slot], (uint32_t)((gc / nslot) & 1), t_step, a.timeout_ns)) {
        if (lane == 0) {
          abort_round(a.sync.hdr, round_s, kStatusTimeout);
          abort_s = 1;
        }
        return false;
      }
      const int ns = ra.ST - c * kChunkStrips;
      if (warp < ns) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        const uint32_t blk = ring_addr + (uint32_t)slot * kChunkBytes +
                             (uint32_t)warp * kSmemStripBytes + (lane >> 3) * 128 + (lane & 7) * 16;
#pragma unroll
        for (int kt = 0; kt < 16; ++kt) {
          uint32_t f0, f1, f2, f3;
          ptx::ldmatrix_x4(blk + kt * 512, f0, f1, f2, f3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            uint32_t b0 = 0u, b1 = 0u;
            if (8 * nt + g < a.B) {
              b0 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + nt) * 128 + lane * 4);
              b1 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + 2 + nt) * 128 + lane * 4);
            }
            ptx::mma_16816(acc[nt], f0, f1, f2, f3, b0, b1);
          }
        }
        logits_strip<NT>(acc, base_s, ra.R, a.B,
                         kTmemRows + 128 * RS + 16 * (ra.S + c * kChunkStrips + warp), lane);
      }
      __syncwarp();
      if (lane == 0) {
        // this warp's reads of the slot are done: order them before the refill
        ptx::fence_proxy_async_smem();
        __threadfence_block();
        if (atomicAdd(&slot_done[slot], 1) == kResWarps - 1) {
          __threadfence_block();
          slot_done[slot] = 0;
          ring_consumed = gc + 1;
          if (gc + nslot < a.gamma * n_chunks) {
            issue_chunk(gc + nslot);
            ring_issued = gc + nslot + 1;
          }
        }
      }
      return true;
    };
    const int c_first = n_chunks < nslot ? n_chunks : nslot;
    bool ring_ok = true;
    for (int c = 0; c < c_first && ring_ok; ++c) ring_ok = consume_chunk(c);

    // (2) register strips and this warp's shared-memory strips (s2 = warp,
    // warp + 8, warp + 16) in ONE k loop: up to RS + SMAX independent mma.sync
    // accumulation chains per warp hide the HMMA latency
    {
      const int nS = (ra.S - warp + kResWarps - 1) / kResWarps;   // this warp's smem strips
      float acc[RS + SMAX][NT][4];
#pragma unroll
      for (int s = 0; s < RS + SMAX; ++s)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[s][nt][e] = 0.0f;
      const uint32_t blk0 = w2_addr + (uint32_t)warp * kSmemStripBytes + (lane >> 3) * 128 +
                            (lane & 7) * 16;
#pragma unroll
      for (int kt = 0; kt < 16; ++kt) {
        uint32_t af[SMAX][4];
#pragma unroll
        for (int j = 0; j < SMAX; ++j)
          if (j < nS)
            ptx::ldmatrix_x4(blk0 + (uint32_t)(j * kResWarps) * kSmemStripBytes + kt * 512,
                             af[j][0], af[j][1], af[j][2], af[j][3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint32_t b0 = 0u, b1 = 0u;
          if (8 * nt + g < a.B) {
            b0 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + nt) * 128 + lane * 4);
            b1 = *reinterpret_cast<const uint32_t*>(U + (4 * kt + 2 + nt) * 128 + lane * 4);
          }
#pragma unroll
          for (int s = 0; s < RS; ++s)
            ptx::mma_16816(acc[s][nt], wr[s][kt][0], wr[s][kt][1], wr[s][kt][2], wr[s][kt][3],
                           b0, b1);
#pragma unroll
          for (int j = 0; j < SMAX; ++j)
            if (j < nS)
              ptx::mma_16816(acc[RS + j][nt], af[j][0], af[j][1], af[j][2], af[j][3], b0, b1);
        }
      }
      trace_stamp(a, k, 1);
#pragma unroll
      for (int s = 0; s < RS; ++s)
        logits_strip<NT>(acc[s], base_s, ra.R, a.B, kTmemRows + (warp * RS + s) * 16, lane);
#pragma unroll
      for (int j = 0; j < SMAX; ++j)
        if (j < nS)
          logits_strip<NT>(acc[RS + j], base_s, ra.R, a.B,
                           kTmemRows + 128 * RS + (warp + j * kResWarps) * 16, lane);
    }

    for (int c = c_first; c < n_chunks && ring_ok; ++c) ring_ok = consume_chunk(c);

    trace_stamp(a, k, 2);

    // (4) tensor-memory rows: warps 0-3 take tiles 0 and 2, warps 4-7 tile 1
    if (a.B == 1) {
      // one request: one column per K half, and a warp's two tiles are read
      // out of tensor memory together (one load latency, not two)
      const int q = warp & 3, t0 = warp >> 2;
      const bool two = t0 == 0;
      bool good = true;
      for (int t = t0; t < kTmemTiles; t += 2)
        good = good && wait_mbar(&mbar[2 * t], (uint32_t)(k & 1), t_step, a.timeout_ns) &&
               wait_mbar(&mbar[2 * t + 1], (uint32_t)(k & 1), t_step, a.timeout_ns);
      if (!good) {
        abort_round(a.sync.hdr, round_s, kStatusTimeout);
        abort_s = 1;
      }
      ptx::tc_fence_after();
      const uint32_t lane_base = (uint32_t)(32 * q) << 16;
      uint32_t d[4][1];
      ptx::tmem_ld<1>(tmem + lane_base + kDCol0 + 32 * t0, d[0]);
      ptx::tmem_ld<1>(tmem + lane_base + kDCol0 + 32 * t0 + 16, d[1]);
      if (two) {
        ptx::tmem_ld<1>(tmem + lane_base + kDCol0 + 64, d[2]);
        ptx::tmem_ld<1>(tmem + lane_base + kDCol0 + 64 + 16, d[3]);
      }
      const int rla = t0 * 128 + 32 * q + lane, rlb = 256 + 32 * q + lane;
      const uint32_t ba = base_s[rla];
      const uint32_t bb = two ? base_s[rlb] : 0u;
      ptx::tmem_wait_ld();
      const float bias_a =
          __bfloat162float(__float2bfloat16_rn(__uint_as_float(d[0][0]) + __uint_as_float(d[1][0])));
      base_s[rla] = float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(ba), bias_a));
      if (two) {
        const float bias_b = __bfloat162float(
            __float2bfloat16_rn(__uint_as_float(d[2][0]) + __uint_as_float(d[3][0])));
        base_s[rlb] = float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(bb), bias_b));
      }
    } else {
      const int q = warp & 3;
#pragma unroll 1
      for (int t = warp >> 2; t < kTmemTiles; t += 2) {
        if (!wait_mbar(&mbar[2 * t], (uint32_t)(k & 1), t_step, a.timeout_ns) ||
            !wait_mbar(&mbar[2 * t + 1], (uint32_t)(k & 1), t_step, a.timeout_ns)) {
          abort_round(a.sync.hdr, round_s, kStatusTimeout);
          abort_s = 1;
        }
        ptx::tc_fence_after();
        uint32_t d0[NCOL], d1[NCOL];
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        ptx::tmem_ld<NCOL>(tmem + lane_base + kDCol0 + 32 * t, d0);        // K half 0
        ptx::tmem_ld<NCOL>(tmem + lane_base + kDCol0 + 32 * t + 16, d1);   // K half 1
        ptx::tmem_wait_ld();
        const int rl = t * 128 + 32 * q + lane;
        uint32_t bvals[NCOL];
#pragma unroll
        for (int c = 0; c < NCOL; ++c) bvals[c] = c < a.B ? base_s[(size_t)c * ra.R + rl] : 0u;
#pragma unroll
        for (int c = 0; c < NCOL; ++c)
          if (c < a.B) {
            const float bias =
                __bfloat162float(__float2bfloat16_rn(__uint_as_float(d0[c]) + __uint_as_float(d1[c])));
            base_s[(size_t)c * ra.R + rl] =
                float_to_bf16_bits_rn(__fadd_rn(bf16_bits_to_float(bvals[c]), bias));
          }
      }
    }
    // (4a) a recurrent head's rows of M @ h_k, released with this step's arrival
    if (CELL && a.cell != 0 && k + 1 < a.gamma) publish_cell_rows(a, U, k, cta, warp, lane, mreg);
    ptx::tc_fence_before();
    __syncthreads();

    // (4b) scores and keys of all rows, every thread
    key_pass<(NT > 1)>(a, base_s, ra.R, nv, row0, k, kpm, eseed, group_best);
    trace_stamp(a, k, 3);
    ptx::tc_fence_before();
    __syncthreads();
    trace_stamp(a, k, 4);

    // (5) next step's base rows (the current ones are no longer read), by
    // warps 1-7: warp 0's release below would otherwise wait for these loads
    if (warp != 0) prefetch_base(ra, k + 1, row0, nv, base_s, 32, kResThreads - 32);

    // (6) the rendezvous (warp 0): per request an atomic max into the step's
    // key slot, released by an arrival count; wait until every CTA has
    // counted every request, read the winners, gather the next u rows
    if (warp == 0) {
      const uint32_t parity = round_s & 1u;
      const uint32_t target = (uint32_t)n_cta;
      uint32_t* cnt = a.sync.count_at(parity, k);
      unsigned long long* keyk = a.sync.key_at(parity, k, 0);
      unsigned long long cand = 0ull;
      if (lane < a.B) {
        unsigned long long mine = 0ull;
        for (int sl = 0; sl < nslots; ++sl) mine = key_max(mine, group_best[lane][sl]);
        if (cta != a.skip_cta) red_relaxed_gpu_max_u64(keyk + lane, mine);
        cand = mine;
      }
      __syncwarp();
      // one arrival per CTA: lane 0's release is cumulative over the maxes the
      // warp barrier ordered before it
      if (lane == 0 && cta != a.skip_cta) red_release_gpu_add(cnt, 1u);
      if (cand != 0ull) {                          // the candidate's W1 row, into L2
        const uint16_t* row = a.W1 + (size_t)(0xFFFFFFFFu - (uint32_t)cand) * kRank;
#pragma unroll
        for (int i = 0; i < 4; ++i) ptx::prefetch_l2(row + 64 * i);
      }
      trace_stamp(a, k, 5);
      int good = 1;
      if (lane == 0) {
        uint32_t spins = 0;
        while (ld_acquire_gpu(cnt) < target) {
          if ((++spins & 63u) == 0u) {
            if (round_aborted(a.sync.hdr, round_s)) { good = 0; break; }
            if ((int64_t)(globaltimer_ns() - t_step) > a.timeout_ns) {
              abort_round(a.sync.hdr, round_s, kStatusTimeout);
              good = 0;
              break;
            }
          }
        }
        if (!good) abort_s = 1;
      }
      good = __shfl_sync(0xFFFFFFFFu, good, 0);
      if (good) {
        trace_stamp(a, k, 6);
        if (lane < a.B) {
          const int32_t tok = key_token(ld_acquire_gpu_u64(keyk + lane));
          if (tok < 0 || (int64_t)tok >= a.V) {    // cannot happen: every CTA posts a real row
            abort_round(a.sync.hdr, round_s, kStatusInternal);
            abort_s = 1;
          } else {
            tok_s[lane] = tok;
            if (cta == 0) a.out_tokens[(size_t)lane * a.gamma + k] = tok;
          }
        }
        __syncwarp();
        // a recurrent head's single request: its next state, here
        // up to four rows: warp 0 fetches them here (larger batches are
        // fetched by all warps after the barrier below)
        for (int b0 = 0; b0 < (a.B <= 4 && !(CELL && a.cell != 0) ? a.B : 0); b0 += 4) {
          uint4 ur[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (b0 + j < a.B)
              ur[j] = __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok_s[b0 + j] * kRank) +
                            lane);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int b = b0 + j;
            if (b < a.B)
              *reinterpret_cast<uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16) = ur[j];
          }
        }
        ptx::fence_proxy_async_smem();
      }
    }
    ptx::cp_async_wait_all();
    ptx::fence_proxy_async_smem();
    __syncthreads();
    if (!(CELL && a.cell != 0) && a.B > 4 && abort_s == 0 && k + 1 < a.gamma) {
      // the next u rows, all in flight at once: warp w fetches rows w, w + 8
      for (int b = warp; b < a.B; b += kResWarps) {
        const uint4 x =
            __ldg(reinterpret_cast<const uint4*>(a.W1 + (size_t)tok_s[b] * kRank) + lane);
        *reinterpret_cast<uint4*>(U + (lane * 2 + (b >> 3)) * 128 + (b & 7) * 16) = x;
      }
      ptx::fence_proxy_async_smem();
      __syncthreads();
    }
    if (CELL && a.cell != 0 && abort_s == 0 && k + 1 < a.gamma) {
      // a recurrent head's next states, every CTA alike, from p (all CTAs'
      // rows of M @ h, read from L2 where the released stores landed), the
      // winner's W1 row and the current state.  One or two requests: thread i
      // updates element i (the gate or tanh of 256 elements side by side);
      // more: warp w updates requests w, w + 8, lane l elements 8l .. 8l + 7
      // (one 16-byte chunk of each operand per lane, fewer round trips)
      if (a.cell == 3 && a.B > 2) {               // the GRU, larger batches: chunk per lane
        for (int b = warp; b < a.B; b += kResWarps) gru_update_row(a, U, k, b, tok_s[b], lane);
      } else if (a.cell == 3) {                   // the GRU: element per thread
        const int i = threadIdx.x;
        for (int b = 0; b < a.B; ++b) {
          const float* pb = a.cell_p + ((size_t)k * 16 + b) * kCellP + i;
          const float pr = __ldcg(pb), pz = __ldcg(pb + kRank), pn = __ldcg(pb + 2 * kRank);
          const uint16_t* xb = a.cell_X + (size_t)tok_s[b] * kRank + i;
          const float xr = bf16_bits_to_float(__ldg(xb));
          const float xz = bf16_bits_to_float(__ldg(xb + (size_t)a.V * kRank));
          const float xn = bf16_bits_to_float(__ldg(xb + (size_t)2 * a.V * kRank));
          uint16_t* hu = u_elem(U, i, b);
          *hu = gru_element(pr, pz, pn, xr, xz, xn, bf16_bits_to_float(*hu));
        }
      } else if (a.B <= 2) {
        const int i = threadIdx.x;
        for (int b = 0; b < a.B; ++b) {
          const float p = ld_relaxed_gpu_f32(a.cell_p + ((size_t)k * 16 + b) * kCellP + i);
          const float x = bf16_bits_to_float(__ldg(a.W1 + (size_t)tok_s[b] * kRank + i));
          uint16_t* hu = u_elem(U, i, b);
          *hu = cell_element(a.cell, p, x, bf16_bits_to_float(*hu));
        }
      } else {
        for (int b = warp; b < a.B; b += kResWarps) cell_update_row(a, U, k, b, tok_s[b], lane);
      }
      ptx::fence_proxy_async_smem();
      __syncthreads();
    }
    trace_stamp(a, k, 7);
    ok = abort_s == 0;
  }

  // -------------------------------------------------------------- exit ----
  ptx::tc_fence_before();
  __syncthreads();
  // a walk that stopped early may leave ring copies in flight: let them land
  // before the CTA's shared memory goes away
  if (threadIdx.x == 0 && ra.ST > 0) {
    const uint64_t t0 = globaltimer_ns();
    for (int gi = ring_consumed; gi < ring_issued; ++gi)
      (void)wait_mbar(&mbar[kMbarRing + gi % nslot], (uint32_t)((gi / nslot) & 1), t0,
                      a.timeout_ns);
  }
  if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
  if (cta == 0) {
    if (!ok)
      for (int i = threadIdx.x; i < a.B * a.gamma; i += blockDim.x) a.out_tokens[i] = -1;
    if (threadIdx.x == 0) atomicAdd(&a.sync.hdr->round, 1u);
  }
}

// Repack row-major W2 [V, 256] into the per-CTA tiered layout (32-bit words,
// each word two consecutive K elements; rows past V are zero), or, with
// `inverse`, write the layout's rows back to row-major form.
__global__ void repack_resident_kernel(uint32_t* __restrict__ W2w, uint32_t* __restrict__ out,
                                       int64_t V, int R, int RS, int64_t words_per_cta,
                                       int n_cta, int inverse) {
  const int64_t total = words_per_cta * n_cta;
  const int64_t rf_words = (int64_t)RS * kRfStripWords;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t cta = i / words_per_cta;
    const int64_t w = i - cta * words_per_cta;
    int rl, kp;
    if (w < kTmemWords) {  // ((((t*2 + h)*16 + c)*4 + q)*32 + l)*4 + ww
      const int ww = (int)(w & 3), l = (int)((w >> 2) & 31), q = (int)((w >> 7) & 3);
      const int c = (int)((w >> 9) & 15), h = (int)((w >> 13) & 1), t = (int)(w >> 14);
      rl = t * 128 + q * 32 + l;
      kp = h * 64 + c * 4 + ww;
    } else if (w < kTmemWords + rf_words) {  // (((ws)*16 + kt)*32 + l)*4 + j, ws = warp*RS + s
      const int64_t x = w - kTmemWords;
      const int j = (int)(x & 3), l = (int)((x >> 2) & 31), kt = (int)((x >> 7) & 15);
      const int ws = (int)(x >> 11);
      rl = kTmemRows + ws * 16 + (l >> 2) + 8 * (j & 1);
      kp = kt * 8 + (l & 3) + 4 * (j >> 1);
    } else {  // ((s2*16 + kt)*4 + m)*32 + i*4 + p
      const int64_t x = w - kTmemWords - rf_words;
      const int p = (int)(x & 3), ii = (int)((x >> 2) & 7), m = (int)((x >> 5) & 3);
      const int kt = (int)((x >> 7) & 15), s2 = (int)(x >> 11);
      rl = kTmemRows + RS * 128 + s2 * 16 + 8 * (m & 1) + ii;
      kp = kt * 8 + 4 * (m >> 1) + p;
    }
    const int64_t row = cta * (int64_t)R + rl;
    if (inverse) {
      if (row < V) W2w[row * (kRank / 2) + kp] = out[i];
    } else {
      out[i] = row < V ? W2w[row * (kRank / 2) + kp] : 0u;
    }
  }
}

}  // namespace

int64_t resident_words_per_cta(int RS, int S) {
  return (int64_t)kTmemWords + (int64_t)RS * kRfStripWords + (int64_t)S * (kSmemStripBytes / 4);
}

int resident_fixed_rows(int RS) { return kTmemRows + 128 * RS; }

int resident_threads() { return kResThreads; }

int resident_max_ring_slots() { return kMaxRingSlots; }

size_t resident_smem_bytes(int S, int ST, int nslot, int max_B, int R) {
  return (size_t)S * kSmemStripBytes + (ST > 0 ? (size_t)nslot * kChunkBytes : 0) +
         16 * 512 + (((size_t)max_B * R * 2 + 15) & ~(size_t)15);
}

const void* resident_kernel_for(int RS, int NT, bool cell) {
  if (RS == 2 && NT == 1 && !cell)
    return reinterpret_cast<const void*>(&walk_resident_kernel<2, 1, 3, false>);
  if (RS == 2 && NT == 2 && !cell)
    return reinterpret_cast<const void*>(&walk_resident_kernel<2, 2, 3, false>);
  if (RS == 2 && NT == 1 && cell)
    return reinterpret_cast<const void*>(&walk_resident_kernel<2, 1, 3, true>);
  if (RS == 2 && NT == 2 && cell)
    return reinterpret_cast<const void*>(&walk_resident_kernel<2, 2, 3, true>);
  return nullptr;
}

int resident_max_smem_strips() { return 3 * kResWarps; }

cudaError_t resident_repack(void* rowmajor, void* packed, int64_t V, int R, int RS, int S,
                            int n_cta, bool inverse, cudaStream_t stream) {
  const int64_t wpc = resident_words_per_cta(RS, S);
  const int64_t total = wpc * n_cta;
  int blocks = (int)((total + 255) / 256);
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  repack_resident_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint32_t*>(rowmajor),
                                                     static_cast<uint32_t*>(packed), V, R, RS, wpc,
                                                     n_cta, inverse ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace dspark
