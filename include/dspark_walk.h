/*
 * dspark_walk.h -- C ABI of the GB300 (sm_103a) serial Markov draft walk.
 *
 * The operation (source: "Keeping the Draft Walk on Chip: One Launch for
 * DSpark's Markov Head", section "The serial part of a parallel drafter"):
 * for every request b, starting from prev = anchor[b], for k = 0 .. gamma-1
 *
 *     u        = W1[prev]                                  (rank r = 256)
 *     bias[v]  = bf16_rne(fp32 sum_j W2[v,j] * u[j])        for every v < V
 *     logit[v] = bf16_rne(fp32(base[b,k,v]) + fp32(bias[v]))
 *     tok      = argmax_v logit[v]              (temperature[b] == 0)
 *              = argmax_v fp32(logit[v] / T) + g(b,k,v)    (T > 0, Gumbel-max)
 *     out_tokens[b,k] = tok;  prev = tok
 *
 * The rounding points are those of section "B200: the bf16 table fits on
 * chip" (fp32 accumulation, bias rounded to bf16, then the sum rounded to
 * bf16).  Ties go to the smallest token id (section "The idea: make the walk
 * resident": the 64-bit key holds the order-preserving logit bits and then
 * the inverted row index).  The Gumbel noise g = -log(-log U) draws U from
 * Philox4x32-10 keyed by (seed, request, step, token): key = (lo32(seed),
 * hi32(seed)), counter = (v >> 2, k, b, 0), token v reads output word v & 3,
 * U = (2 * (x >> 9) + 1) * 2^-24.  All of it is computed in fp32.
 *
 * One round is ONE persistent kernel launch on the caller's stream; every
 * step of the walk runs inside it and only token ids cross between steps
 * (same section).  All CTAs are co-resident (cooperative launch).
 *
 * Conventions for every call:
 *  - Return value 0 (DSPARK_OK) or a negative DSPARK_E* code.  Nothing traps.
 *  - "device" pointers are CUDA device (or managed) memory of the current
 *    device; "host" pointers are ordinary or pinned host memory.
 *  - bf16 arrays are IEEE bfloat16 bit patterns, 2 bytes per element,
 *    row-major and contiguous.
 *  - `stream` is a cudaStream_t (0 = the legacy default stream).
 *  - Calls on one handle must be ordered by the caller (one stream, or
 *    streams joined by events), as for a CUDA graph.
 */
#ifndef DSPARK_WALK_H
#define DSPARK_WALK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define DSPARK_OK 0
#define DSPARK_EINVAL (-1)       /* bad argument, detected on the host before launch */
#define DSPARK_ENOMEM (-2)       /* device allocation failed in create */
#define DSPARK_ECUDA (-3)        /* a CUDA runtime call failed */
#define DSPARK_ETIMEOUT (-4)     /* a cross-CTA rendezvous waited past its limit */
#define DSPARK_EANCHOR (-5)      /* an anchor was outside [0, V) (device-detected) */
#define DSPARK_EUNSUPPORTED (-6) /* r != 256, or the device is not sm_103 */
#define DSPARK_ETEMP (-7)        /* a temperature was negative or not finite (device-detected) */
#define DSPARK_ELIMIT (-8)       /* B or gamma above dspark_walk_run_noalloc's fixed maximum */
#define DSPARK_EINTERNAL (-9)    /* a device-side consistency check failed (a bug; tokens -1) */

/* Opaque handle: resident weight layout, rendezvous slots, status word. */
typedef struct dspark_walk dspark_walk;
typedef dspark_walk *dspark_walk_t;

/*
 * How create() placed W2 on the chip (see dspark_walk_get_plan).
 * Rows of W2 are split into contiguous per-CTA shards; inside a shard each
 * row lives in exactly one tier.
 */
struct dspark_walk_plan {
    int64_t V;              /* vocabulary size */
    int r;                  /* rank (256) */
    int n_cta;              /* CTAs of the persistent kernel (one per SM used) */
    int threads;            /* threads per CTA */
    int rows_per_cta;       /* rows of the largest shard */
    int rows_tmem;          /* per CTA: rows held in tensor memory */
    int rows_smem;          /* per CTA: rows held in shared memory */
    int rows_rf;            /* per CTA: rows held in registers */
    int rows_stream;        /* per CTA: rows re-read from L2/HBM every step */
    int64_t resident_bytes; /* W2 bytes held on chip across steps, all CTAs */
    int64_t streamed_bytes; /* W2 bytes re-read from L2/HBM per step, all CTAs */
    int max_B;              /* largest batch a run may pass */
    int max_gamma;          /* longest walk a run may pass */
    int kernel;             /* which kernel runs small batches (DSPARK_KERNEL_*) */
    int sm_count;           /* SMs on the device */
    int64_t weight_bytes;   /* device bytes of the W2 layouts the handle holds now */
};

#define DSPARK_KERNEL_STREAM 0   /* every row re-read from global memory each step */
#define DSPARK_KERNEL_RESIDENT 1 /* rows held in registers / shared / tensor memory */
#define DSPARK_KERNEL_BATCHED 2  /* rows streamed by TMA, tcgen05 with N = B (large B) */

/*
 * dspark_walk_create -- prepare a walk over fixed weights ("Keeping the Draft
 * Walk on Chip", section "The idea: make the walk resident": the weights are
 * laid out once so that each CTA can load its slice of W2 rows at the start
 * of a round; section "B200: the bf16 table fits on chip" for the split of
 * those rows over tensor memory, shared memory and registers).
 *
 *   W1        device, bf16 [V, r] row-major: the Markov embedding.  Referenced,
 *             not copied: keep it alive and unchanged until destroy.
 *   W2        device, bf16 [V, r] row-major: the vocabulary projection.
 *             Copied and repacked into a handle-owned layout (V * r * 2
 *             bytes); the caller may free it after create returns.
 *   V         1 <= V < 2^31
 *   r         must be 256 (DSPARK_EUNSUPPORTED otherwise)
 *   max_B     1 <= max_B <= 256: largest batch any run will pass
 *   max_gamma 1 <= max_gamma <= 64: longest walk any run will pass
 *   out       receives the handle (set to NULL on failure)
 *
 * The handle holds W2 only in the layouts its runs can take under its current
 * settings (the on-chip layout of the resident kernels, and the batched
 * kernel's layout when max_B is above the resident batch); another layout is
 * built from one it holds when set_kernel / set_cell / set_state_output first
 * need it.  dspark_walk_get_plan reports the bytes held (weight_bytes).
 * Uses the current CUDA device; synchronises it once.  Errors: DSPARK_EINVAL,
 * DSPARK_EUNSUPPORTED, DSPARK_ENOMEM, DSPARK_ECUDA.
 */
int dspark_walk_create(const void *W1, const void *W2, int64_t V, int r, int max_B,
                       int max_gamma, dspark_walk_t *out);

/*
 * dspark_walk_run -- one round: the whole gamma-step walk for B requests in
 * one launch on `stream` (asynchronous; capturable in a CUDA graph, and needs
 * no memset between replays: the rendezvous state alternates by round parity).
 * Source: "Keeping the Draft Walk on Chip", section "The serial part of a
 * parallel drafter" (the recurrence), section "The idea: make the walk
 * resident" (one launch per round, the cross-CTA selection, per-request
 * temperatures read on the device, logits written for the verifier).
 *
 *   base_logits  device, bf16 [B, gamma, V]: the parallel pass's logits
 *   anchor       device, int32 [B]: the last accepted token of each request
 *   temperature  device, fp32 [B]: 0 = greedy, > 0 = Gumbel-max sampling.
 *                fp32(logit / T) is the product with fl(1/T), within one
 *                fp32 ulp of the quotient, and overflows to +-inf where the
 *                quotient does (then the smallest such token id wins).
 *                Under the group sampler a request whose logit / T
 *                overflows fp32 draws a valid but unspecified token.
 *   seed         Philox key of this round (change it per round for fresh noise)
 *   out_tokens   device, int32 [B, gamma]: the drafted tokens
 *   B, gamma     1 <= B <= max_B, 1 <= gamma <= max_gamma
 *   out_logits   NULL, or device bf16 [B, gamma, V]: receives every logit the
 *                tokens were chosen from (for a lossless verifier)
 *
 * Host-detectable errors (NULL pointers, sizes) return DSPARK_EINVAL before
 * any launch.  Device-detected errors (anchor out of range, bad temperature,
 * rendezvous timeout) set the handle's status word and write -1 to
 * out_tokens; read them with dspark_walk_status.
 */
int dspark_walk_run(dspark_walk_t h, const void *base_logits, const int32_t *anchor,
                    const float *temperature, uint64_t seed, int32_t *out_tokens, int B,
                    int gamma, void *out_logits, void *stream);

/*
 * dspark_walk_run_host -- the same round with HOST buffers, then waits for
 * `stream`.  Anchor and temperature go through a pinned block the handle
 * owns, which the kernel reads in place.  Base logits in pinned host memory
 * (cudaHostAlloc / cudaHostRegister / a pinned PyTorch tensor) of at most
 * 16 MiB are read in place by the kernel over the host link, each CTA
 * fetching its rows one step ahead; other base buffers are first copied to
 * a handle-owned device buffer on `stream`.  Tokens go straight into a pinned
 * out_tokens_host, otherwise through a device buffer and a copy; logits (if
 * out_logits_host is not NULL) always through a device buffer and a copy.
 * The round's status comes back on the same stream, so the call synchronises
 * once.  Returns the round's device status (as dspark_walk_status does, and
 * clears it) or a host-side error.  Host buffers must not change until the
 * call returns.
 */
int dspark_walk_run_host(dspark_walk_t h, const void *base_logits_host,
                         const int32_t *anchor_host, const float *temperature_host,
                         uint64_t seed, int32_t *out_tokens_host, int B, int gamma,
                         void *out_logits_host, void *stream);

/*
 * dspark_walk_status -- wait for `stream`, then return and clear the status
 * word the device wrote during earlier runs (DSPARK_OK if none failed).  The
 * pages define no error channel; device-detected errors (a bad anchor or
 * temperature, a rendezvous timeout) set this word instead of trapping.
 */
int dspark_walk_status(dspark_walk_t h, void *stream);

/*
 * dspark_walk_get_plan -- copy the placement chosen at create into *p (the
 * per-CTA split of W2 rows over the on-chip tiers: "Keeping the Draft Walk on
 * Chip", sections "B200: the bf16 table fits on chip" and "V = 248,320: 62% on
 * chip, the rest streamed"), with the bytes of W2 layouts held now.
 */
int dspark_walk_get_plan(dspark_walk_t h, struct dspark_walk_plan *p);

/*
 * dspark_walk_set_limits -- rendezvous wait limit in nanoseconds (default
 * 200,000,000; minimum 1,000) and a fault-injection switch: skip_cta >= 0
 * makes that CTA skip posting its arrival, so every other CTA's wait runs
 * out and the round ends with DSPARK_ETIMEOUT (tests use it to check that a
 * lost arrival is reported, not hung on).  skip_cta = -1 turns it off.
 * Takes effect from the next run.
 */
int dspark_walk_set_limits(dspark_walk_t h, int64_t timeout_ns, int skip_cta);

/*
 * dspark_walk_set_kernel -- choose the kernels of later runs.
 *   DSPARK_KERNEL_RESIDENT (default): the resident kernel for batches up to
 *     its limit (when create() found an on-chip placement), the batched
 *     kernel above it.  DSPARK_EUNSUPPORTED if no resident placement exists.
 *   DSPARK_KERNEL_BATCHED: the batched kernel for every batch.
 *   DSPARK_KERNEL_STREAM: the CUDA-core kernel that re-reads W2 from L2/HBM
 *     every step (the single-launch "L2 probe" of the blog post's section
 *     "V = 151,936: the whole bf16 table on chip"), kept as an ablation.
 */
int dspark_walk_set_kernel(dspark_walk_t h, int kernel);

/*
 * dspark_walk_set_seed_mode -- how later runs key their Philox noise.
 *   DSPARK_SEED_FIXED (default): the key is `seed` as passed to the run.
 *   DSPARK_SEED_PER_ROUND: the key is seed + n (mod 2^64), n = the number of
 *     rounds this handle has run before (0 for the first run after create;
 *     rounds rejected by the host checks do not count; rounds the kernel ends
 *     with an error status do).  The pages key the noise on the seed and a
 *     round counter ("Keeping the Draft Walk on Chip...", section "The idea:
 *     make the walk resident"); with this mode one CUDA graph captured with a
 *     fixed seed draws fresh noise on every replay, with no host update.
 * DSPARK_EINVAL for another mode.
 */
#define DSPARK_SEED_FIXED 0
#define DSPARK_SEED_PER_ROUND 1
int dspark_walk_set_seed_mode(dspark_walk_t h, int mode);

/*
 * dspark_walk_set_sampler -- how later runs sample requests with T > 0.
 *   DSPARK_SAMPLER_GUMBEL (default): per-token Gumbel-max, every token's score
 *     fp32(logit / T) - log(-log U) with U from Philox counter (v >> 2, k, b, 0)
 *     word v & 3 ("Keeping the Draft Walk on Chip...", section "The idea: make
 *     the walk resident").
 *   DSPARK_SAMPLER_GROUP: the same page's large-batch sampler, an inverse CDF
 *     inside groups of 8 consecutive tokens and Gumbel-max across the groups,
 *     with vLLM pull request #64442's in-group step (section "Details"): for
 *     group j, z = logit / T, m = max z, weights exp(z - m) of mass S; group
 *     score m + log S - log(-log U1); inside the winning group the first token
 *     whose running sum of weights exceeds U2 * S.  U1, U2 are words 2 (j & 1)
 *     and 2 (j & 1) + 1 of Philox counter (j >> 1, k, b, 1).  Tokens follow
 *     softmax(logit / T) as under Gumbel-max, but they are other draws; T = 0
 *     requests are greedy either way.  One Philox call serves 16 tokens and each
 *     token costs one exp instead of two logs.  Runs that would take the
 *     streamed kernel (DSPARK_KERNEL_STREAM) return DSPARK_EUNSUPPORTED.
 * DSPARK_EINVAL for another value.
 */
#define DSPARK_SAMPLER_GUMBEL 0
#define DSPARK_SAMPLER_GROUP 1
int dspark_walk_set_sampler(dspark_walk_t h, int sampler);

/*
 * dspark_walk_set_cell -- which serial head later runs walk ("Keeping the Draft
 * Walk on Chip", section "Beyond DSpark: other serial heads": the walk as a
 * template over the head's state update).
 *   DSPARK_CELL_MARKOV (default): u_k = W1[prev_k]; M and X are ignored.
 *   DSPARK_CELL_GATED, DSPARK_CELL_RNN: a recurrent head with state h (256
 *     bf16 values per request), h_{-1} = 0, x_k = W1[prev_k] (prev_0 = the
 *     anchor), p = M @ h_{k-1} accumulated in fp32, and per element
 *       gated: z = 1 / (1 + exp(-p)), h_k = bf16((1 - z) h_{k-1} + z x_k)
 *       RNN:   h_k = bf16(tanh(p + x_k))
 *     M: device bf16 [256, 256] row-major.
 *   DSPARK_CELL_GRU: the page's GRU heads, with the input projections folded
 *     into three token tables X = (X_r, X_z, X_n), device bf16 [3, V, 256], and
 *     M = (M_r; M_z; M_n) stacked, device bf16 [768, 256]: with p_g = M_g @ h_{k-1},
 *       r = sig(X_r[prev_k] + p_r), z = sig(X_z[prev_k] + p_z),
 *       n = tanh(X_n[prev_k] + r p_n), h_k = bf16((1 - z) n + z h_{k-1})
 *     (W1 is not read by this head).
 *   All in fp32, each operation rounded; u_k = h_k is projected through W2 and
 *   selected from exactly as W1[prev] is.  The pages print no cell equations:
 *   these are the plain gated, Elman and GRU forms.
 *   M and X are 16-byte aligned and referenced (not copied): the caller keeps
 *   them alive and unchanged while runs use them.
 *   Each CTA computes its share of the recurrent rows for every request and
 *   publishes them with its arrival at the step's rendezvous; after the
 *   rendezvous every CTA forms the new state itself, so a recurrent step adds
 *   no exchange.  Recurrent runs take the resident kernel (B <= the handle's
 *   resident batch, at most 16); other runs return DSPARK_EUNSUPPORTED, as does
 *   this call on a handle without a resident layout (V >= 2^18).  DSPARK_EINVAL
 *   for another cell, a null or misaligned M (or X for the GRU);
 *   DSPARK_ENOMEM / DSPARK_ECUDA if the 48 KB per step of exchange memory
 *   cannot be allocated (first recurrent cell only).
 */
#define DSPARK_CELL_MARKOV 0
#define DSPARK_CELL_GATED 1
#define DSPARK_CELL_RNN 2
#define DSPARK_CELL_GRU 3
int dspark_walk_set_cell(dspark_walk_t h, int cell, const void *M, const void *X);

/*
 * dspark_walk_set_state_output -- where later runs write each step's latent
 * u_k (the recurrent state h_k, or W1[prev_k] for the Markov head): device
 * bf16 [B, gamma, 256], caller-owned; NULL (the default) writes nothing.
 * Only the resident kernel writes it; runs that would take another kernel
 * return DSPARK_EUNSUPPORTED while it is set.  DSPARK_EINVAL if misaligned.
 */
int dspark_walk_set_state_output(dspark_walk_t h, void *out_state);

/*
 * dspark_walk_round -- the handle's round counter n (see set_seed_mode):
 * synchronises `stream` (a cudaStream_t; NULL = legacy default stream), then
 * reads it into *round.
 */
int dspark_walk_round(dspark_walk_t h, void *stream, uint64_t *round);

/*
 * dspark_walk_gumbel_noise -- the Gumbel noise the kernels add to logit / T:
 * noise[i] = g(bits[i]), g = -log(-log U), U = (2 (bits >> 9) + 1) 2^-24 (the
 * uniform of a Philox output word), in the kernels' own fp32 arithmetic.  It
 * exists so that the noise can be checked against a float64 reference over
 * every uniform (the pages fix the formula, not its implementation).
 *   bits, noise  device, n uint32 / n float32
 * Asynchronous on `stream`; DSPARK_EINVAL for n < 0 or null pointers with n > 0.
 */
int dspark_walk_gumbel_noise(const uint32_t *bits, float *noise, int64_t n, void *stream);

/*
 * dspark_walk_set_trace -- phase timing of later runs (profiling aid).  When
 * `device_buffer` holds at least n_cta * (gamma + 1) * 8 uint64 values, each
 * run's CTA c writes SM clock64() stamps of its thread 0 at
 * [(c * (gamma + 1) + slot) * 8 + phase]: slot k < gamma is step k (stamps:
 * 0 start, 1 projection k loop issued, 2 epilogue done (keys, or logits),
 * 3 key pass done, 4 CTA barrier passed, 5 key posted, 6 winner seen,
 * 7 next u gathered; the tcgen05 resident kernel stamps 1 after its register
 * strips, 2 after its shared strips, 3 after its tensor-memory epilogue and
 * key pass); slot gamma is the round's entry (0 start, 1 tensor-memory and
 * register tiers loaded, 2 ready; the mma.sync kernel also stamps 3 at the
 * CTA's first instruction and 4 at its last).  Only the resident kernels
 * write stamps.
 * NULL turns tracing off.
 */
int dspark_walk_set_trace(dspark_walk_t h, void *device_buffer, int64_t bytes);

/*
 * dspark_walk_set_trace_clock -- what later traced runs stamp:
 *   DSPARK_TRACE_SM_CLOCK (default): clock64() cycles of the CTA's SM (fine
 *     grained; not comparable between SMs);
 *   DSPARK_TRACE_GLOBAL_TIMER: the global timer in nanoseconds (coarser, but
 *     one clock for every SM, so the CTAs' stamps of one step can be compared:
 *     how far apart they post their keys and see the winner).
 * DSPARK_EINVAL for another value.
 */
#define DSPARK_TRACE_SM_CLOCK 0
#define DSPARK_TRACE_GLOBAL_TIMER 1
int dspark_walk_set_trace_clock(dspark_walk_t h, int clock);

/*
 * dspark_walk_unit_rates -- measure, on the current device, the rates at
 * which the resident walk's on-chip tiers feed the tensor cores: the unit
 * costs of the walk's on-chip-read roofline ("Keeping the Draft Walk on
 * Chip", section "B200: the bf16 table fits on chip": tcgen05 reads the
 * tensor-memory part of W2, mma.sync the register and shared-memory parts).
 * One CTA of 256 threads per SM runs each pattern; the medians over SMs are
 * written to out (SM clock cycles):
 *   out[0]  mma.sync m16n8k16 bf16, A in registers: cycles per MMA per SM
 *   out[1]  mma.sync with A read by ldmatrix from shared memory: per MMA
 *   out[2]  tcgen05.mma M=128 N=16 K=16, A in tensor memory, six issuing
 *           warps: cycles per MMA per SM
 *   out[3]  one step's projection at the resident shapes (48 tensor-memory
 *           MMAs, 16 k-tiles of 2 register and 3 shared strips per warp)
 *   out[4]  SM clock during the probe, MHz (clock64 over the global timer)
 *   out[5]  tcgen05.ld of 32-column blocks: cycles per KB per SM (n_out >= 7)
 *   out[6]  one step's projection with 4 tensor-memory strips per warp fed to
 *           mma.sync by tcgen05.ld, 1 register and 3 shared strips (n_out >= 7)
 *   out[7]  (input, n_out >= 8) nonzero: random MMA operands, else constant
 *   out[8]  one cross-SM hop: ns from one SM's relaxed store until another
 *           SM's poll sees it, median over five SM pairs (n_out >= 10)
 *   out[9]  one dependent load that hits in L2: cycles (n_out >= 10)
 * n_out >= 5.  Allocates and frees a few KB of device memory, runs on
 * `stream` and synchronises it.  DSPARK_EINVAL (out NULL or n_out < 5),
 * DSPARK_EUNSUPPORTED (not sm_103), DSPARK_ENOMEM, DSPARK_ECUDA, and
 * DSPARK_ETIMEOUT if a tensor-core completion wait ran out.
 */
int dspark_walk_unit_rates(double *out, int n_out, void *stream);

/* dspark_walk_strerror -- a static description of a status code. */
const char *dspark_walk_strerror(int code);

/*
 * dspark_walk_destroy -- free everything the handle owns (the W2 layouts
 * dspark_walk_create built, the rendezvous memory, the staging buffers);
 * synchronises the device.  W1 and any M / X passed to set_cell stay the
 * caller's.
 */
int dspark_walk_destroy(dspark_walk_t h);

/*
 * dspark_walk_run_noalloc -- one round of the walk that allocates no device
 * memory at all (the pages have no counterpart; it exists for callers, not
 * for the method).  Some callers may not call cudaMalloc: code running inside
 * a memory allocator or its callbacks, processes whose device memory belongs
 * to a caching pool that must not be bypassed, and latency-critical paths
 * that must never wait on the driver's allocator.  They cannot use
 * dspark_walk_create, which allocates.
 *
 *   W1, W2       device, bf16 [V, r] row-major (read in place every step:
 *                this is the streamed kernel, no on-chip residency)
 *   other arguments as dspark_walk_run; 1 <= B <= 64, 1 <= gamma <= 16
 *                (DSPARK_ELIMIT above that)
 *
 * The rendezvous slots live in one fixed ~17.5 KB block of device memory
 * built into the library (every GPU that loads the library keeps it until
 * the process exits).  The block's address belongs to a CUDA context: every
 * call looks it up in the caller's current context (cudaGetSymbolAddress, a
 * lookup that allocates nothing) and makes sure the kernels it launches are
 * loaded, so the entry point also works in a context created after
 * cudaDeviceReset.  The first call in a context is where the driver loads
 * those kernels (with lazy module loading that may allocate and synchronise):
 * make it once before capturing a stream into a CUDA graph or entering code
 * that must not allocate.  Each call clears the block on `stream` before its
 * launch; calls that could overlap on the GPU (unordered streams) race on the
 * block and must not be made.  Device-detected errors (bad anchor or
 * temperature, a rendezvous timeout) are reported only as -1 in out_tokens.
 */
int dspark_walk_run_noalloc(const void *W1, const void *W2, int64_t V, int r,
                            const void *base_logits, const int32_t *anchor,
                            const float *temperature, uint64_t seed, int32_t *out_tokens, int B,
                            int gamma, void *out_logits, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_WALK_H */
