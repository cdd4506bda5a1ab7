/*
 * psgd.h — C ABI of the GB300 PowerSGD gradient-compression step (libpsgd.so).
 *
 * One call of psgd_step runs, for every weight-gradient matrix j of every resblock b
 * and every simulated data-parallel worker w held on this GPU:
 *
 *   g_w   = G_w * (1/s_b); nonfinite entries of g_w set to 0 and counted
 *   M_w   = round_E(g_w + E_w)                       (E_w: the error buffer)
 *   skip_b = (nonfinite count of block b over all workers >= threshold_b)
 *   P     = (1/W) sum_w M_w Q                        (first exchange point)
 *   P^    = orthonormal basis of span(P)             (fp32, shifted CholeskyQR)
 *   Q     = (1/W) sum_w M_w^T P^                     (second exchange point; new Q state)
 *   G^    = P^ Q^T                                   (fp32-accurate products)
 *   E_w   = round_E(M_w - G^)
 *   gains/biases: u = (1/W) sum_w zero_nonfinite(U_w * (1/s_b)) in fp32
 *
 * Sources for what each step computes:
 *   "Zero-Shot Text-to-Image Generation - 中文验证版" (reading card), §方法适配: per-
 *     resblock gradient scales; PowerSGD all-reduces low-rank factors; total rank 896
 *     = 112 per GPU shard; embedding/unembedding/gains/biases reduced in 32-bit.
 *     §证据: error buffer, finiteness checks, grouped all-reduce, 32-bit products for
 *     the decompressed gradient.
 *   "[논문 정리] Zero-Shot Text-to-Image Generation", §Mixed-Precision Training: unscale
 *     when the block ends, and Inf/NaN are set to 0. PowerSGD list: the gradient is
 *     accumulated into the error buffer, and gains/biases stay uncompressed in 32-bit.
 *   "AIGC 基本功|混合精度与数值稳定性", §6.2: every data-parallel rank takes the same
 *     skip decision.
 *
 * Conventions (all entry points):
 *   - Every device pointer is owned by the caller. The library allocates no device
 *     memory. Its scratch lives in the caller's workspace (psgd_workspace_size). The
 *     handle owns only host-side plans and one pinned host staging buffer.
 *   - Matrices are row-major and dense: leading dimension = n. Device pointers to
 *     gradients, error buffers and G^ must be 16-byte aligned, and n * element size
 *     must be a multiple of 16 bytes.
 *   - Nothing throws or exits across the ABI. Argument errors return PSGD_EINVAL or
 *     PSGD_EUNSUPPORTED before any launch. CUDA launch/runtime errors return
 *     PSGD_ECUDA. psgd_last_error() returns a per-thread message for the last failure.
 *   - psgd_step is asynchronous on `stream` (a cudaStream_t, or NULL for the legacy
 *     default stream). The handle keeps the last 4 distinct pointer/scale tables (with
 *     the TMA descriptors of their G and E buffers) on the device, so buffer sets used
 *     in turn are encoded and uploaded once. A table that is none of those replaces the
 *     least recently used one; the host then waits only if that slot's own upload, 4
 *     tables ago, has not finished. Calls on one handle must be ordered on the device
 *     (one stream, or streams joined by events): a table is overwritten in stream order.
 */
#ifndef PSGD_H_
#define PSGD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PSGD_F32 = 0, PSGD_F16 = 1, PSGD_BF16 = 2 } psgd_dtype;

typedef enum {
  PSGD_OK = 0,
  PSGD_EINVAL = 1,        /* bad argument: null pointer, bad shape, misalignment, ... */
  PSGD_ECUDA = 2,         /* a CUDA runtime or launch error */
  PSGD_EUNSUPPORTED = 3,  /* valid but not supported by this library (e.g. dtype mix) */
  PSGD_ETIMEOUT = 4       /* a bounded device-side wait expired (see psgd_check) */
} psgd_status;

typedef struct {
  int64_t m, n; /* rows, columns of one weight-gradient matrix */
} psgd_shape;

/* Flags (psgd_config.flags). */
#define PSGD_FLAG_SIMT 0x1u          /* use the FFMA GEMM engine for 16-bit too (debug) */
#define PSGD_FLAG_MASK 0x2u          /* write the nonfinite mask bitmap (debug output) */
#define PSGD_FLAG_STOP_AFTER_INGEST 0x4u /* only unscale/mask/count/M and skip (debug) */
#define PSGD_FLAG_DEBUG_EXPIRE_WAIT 0x8u /* test of the bounded waits (tensor engine only):
                                            every CTA of the decompression kernel waits a
                                            few hundred microseconds on a barrier that
                                            nothing completes, then winds down. The step's
                                            G^, E and Q are invalid, and psgd_check returns
                                            PSGD_ETIMEOUT. */
#define PSGD_FLAG_EXCHANGE 0x10u     /* plan the data-parallel exchange points: workspace
                                        for the P and Q exchange buffers, and the calls
                                        psgd_step_p / psgd_step_q / psgd_step_e. Needs
                                        unc_len == 0 and not STOP_AFTER_INGEST. */

typedef struct {
  int32_t num_blocks;       /* B >= 1 resblocks */
  int32_t mats_per_block;   /* J >= 1 matrices per resblock */
  int32_t num_workers;      /* W >= 1 simulated data-parallel workers */
  int32_t rank;             /* r, 1 <= r <= min(m, n) for every matrix */
  const psgd_shape* shapes; /* [J] host array: every block has the same J shapes */
  int32_t grad_dtype;       /* psgd_dtype of G */
  int32_t err_dtype;        /* psgd_dtype of E (and of M). 16-bit G needs the same
                               16-bit E; fp32 G needs fp32 E. */
  int64_t unc_len;          /* fp32 gains+biases per block per worker (0 = none) */
  double skip_fraction;     /* T in (0, 1]: skip block b when its nonfinite count over
                               all workers is >= ceil(T * W * numel_b) (IEEE double) */
  uint32_t flags;           /* PSGD_FLAG_* */
} psgd_config;

typedef struct psgd_handle psgd_handle;

/* Arguments of one step. Host arrays of device pointers, indexed as stated. */
typedef struct {
  const void* const* grads;     /* [B*J*W] G_{b,j,w} at ((b*J)+j)*W+w, grad_dtype m x n */
  void* const* errs;            /* [B*J*W] E_{b,j,w}, err_dtype m x n, read and updated */
  float* const* q_state;        /* [B*J] Q_{b,j}, fp32 n x r row-major; the caller
                                   writes Q0 before the first step; updated in place */
  const float* scales;          /* [B] host: s_b, finite and > 0 (powers of two give
                                   a bit-exact M). Below 1, 1/s_b > 1 and a product
                                   that overflows counts as nonfinite, as for device
                                   scales. May be NULL when scales_device is given;
                                   ignored then. */
  float* const* ghat;           /* [B*J] G^_{b,j}, fp32 m x n (written; 0 when skipped) */
  const float* const* unc_in;   /* [B*W] raw gains/biases, fp32 unc_len (NULL if none) */
  float* const* unc_out;        /* [B] mean gains/biases, fp32 unc_len (NULL if none) */
  int64_t* counts;              /* device [B*W]: nonfinite entries of block b, worker w
                                   (matrices and gains/biases); overwritten each step */
  uint8_t* skip;                /* device [B]: 1 when block b was skipped */
  uint32_t* mask_bits;          /* device, only with PSGD_FLAG_MASK (else ignored): one
                                   bit per matrix entry, LSB-first in 32-bit words,
                                   row-major; matrix (b,j,w) starts at word
                                   psgd_mask_offset(cfg, b, j, w). Bits past a matrix's
                                   last entry in its last word are unspecified. */
  const float* scales_device;   /* [B] device, or NULL: s_b read on the device (the state
                                   psgd_scale_update keeps), so no host round trip sits
                                   between steps. Each s_b must be > 0; it may be below 1
                                   (then 1/s_b > 1, and a product that overflows counts
                                   as nonfinite). Nothing checks the values on the host;
                                   psgd_scale_update keeps them finite normal floats. */
} psgd_step_args;

/* Bytes of device workspace psgd_init needs for this configuration (0 on error). */
size_t psgd_workspace_size(const psgd_config* cfg);

/* Word offset of matrix (b, j, w) in the mask bitmap, and the bitmap's total words. */
int64_t psgd_mask_offset(const psgd_config* cfg, int32_t b, int32_t j, int32_t w);
int64_t psgd_mask_words(const psgd_config* cfg);

/* Validate cfg and plan the step into `workspace` (device, >= psgd_workspace_size
 * bytes, 256-byte aligned, owned by the caller, alive until psgd_finalize). On
 * PSGD_OK *out holds a handle. Work is enqueued on `stream` (workspace clearing). */
psgd_status psgd_init(const psgd_config* cfg, void* workspace, size_t ws_bytes,
                      void* stream, psgd_handle** out);

/* Enqueue one PowerSGD step on `stream` (see the top of this file). */
psgd_status psgd_step(psgd_handle* h, const psgd_step_args* args, void* stream);

/* Data-parallel exchange points (a handle made with PSGD_FLAG_EXCHANGE).
 *
 * The method all-reduces the two low-rank factors between machines instead of the
 * gradient ("Zero-Shot Text-to-Image Generation - 中文验证版", §方法适配), and every rank
 * takes the same skip decision ("AIGC 基本功|混合精度与数值稳定性", §6.2). With R ranks
 * (one handle each, W workers per rank; W may differ between ranks, total_workers =
 * the sum), one step is three calls with two caller all-reduces (sum) between them:
 *
 *   psgd_step_p(h, args, s)      ingest, nonfinite counts, and this rank's sum
 *                                P_r = sum_w M_w Q into psgd_exchange_p(h, b, j)
 *                                (fp32 m x r, row-major), and the rank's per-block
 *                                nonfinite counts into psgd_exchange_counts(h) (int64 [B]).
 *   caller: all-reduce (sum) every exchange P buffer and the counts over the ranks.
 *   psgd_step_q(h, args, counts, total_workers, s)
 *                                skip_b from the summed counts, P = sum / total_workers,
 *                                orthonormalisation, and this rank's sum Q_r = sum_w
 *                                M_w^T P^ into psgd_exchange_q(h, b, j) (fp32 n x r).
 *   caller: all-reduce (sum) every exchange Q buffer.
 *   psgd_step_e(h, args, total_workers, s)
 *                                Q state = sum / total_workers, G^ and the error update.
 *
 * All three calls take the same psgd_step_args as psgd_step (the same tables; the skip
 * flags are written by psgd_step_q). Every rank must hold the same Q state at the start
 * of a step (the previous step's all-reduced Q). Skipped blocks leave their buffers
 * untouched in the later calls; the caller may still all-reduce them. The sums are
 * fp32 round-to-nearest; an all-reduce that adds in another order changes the low bits
 * of P and Q, not the method. With one rank (the buffers passed through unchanged) the
 * three calls give bit for bit the result of psgd_step.
 * block_counts: device int64 [B], 8-byte aligned: the per-block nonfinite counts summed
 * over every rank (it may be the psgd_exchange_counts buffer itself, all-reduced in place).
 * total_workers >= this handle's num_workers. Errors: PSGD_EUNSUPPORTED without the flag,
 * PSGD_EINVAL for a bad pointer or total_workers, as for psgd_step otherwise. */
psgd_status psgd_step_p(psgd_handle* h, const psgd_step_args* args, void* stream);
psgd_status psgd_step_q(psgd_handle* h, const psgd_step_args* args, const int64_t* block_counts,
                        int32_t total_workers, void* stream);
psgd_status psgd_step_e(psgd_handle* h, const psgd_step_args* args, int32_t total_workers,
                        void* stream);
/* Device addresses of the exchange buffers (inside the workspace; valid while the handle
 * lives), or NULL for a handle without PSGD_FLAG_EXCHANGE or an index out of range.
 * The P buffers of all matrices lie back to back in (b, j) order, fp32 m_j x r each, so
 * one all-reduce of B * sum_j m_j * r floats from psgd_exchange_p(h, 0, 0) covers them;
 * likewise the Q buffers (B * sum_j n_j * r floats from psgd_exchange_q(h, 0, 0)).
 * psgd_exchange_counts: int64 [B], written by psgd_step_p. */
float* psgd_exchange_p(psgd_handle* h, int32_t b, int32_t j);
float* psgd_exchange_q(psgd_handle* h, int32_t b, int32_t j);
int64_t* psgd_exchange_counts(psgd_handle* h);

/* Dynamic per-resblock gradient scale ("AIGC 基本功|混合精度与数值稳定性", §3.2, the
 * dynamic scaler rule, applied per resblock as "Zero-Shot Text-to-Image Generation -
 * 中文验证版" §方法适配 gives each resblock its own scale). From the nonfinite counts a
 * finished psgd_step left in `counts`, for every block b:
 *   if sum_w counts[b*W + w] > 0:  scale[b] = fp32(scale[b] * fp32(backoff)), streak[b] = 0
 *   else: streak[b] += 1; if streak[b] >= interval:
 *                                   scale[b] = fp32(scale[b] * fp32(growth)), streak[b] = 0
 *   num_blocks  B >= 1, num_workers W >= 1
 *   counts      device int64 [B*W] (psgd_step's counts), read
 *   scale       device fp32 [B], read and written (pass it to the next step as
 *               psgd_step_args.scales_device)
 *   streak      device int32 [B], read and written; the caller starts it at 0
 *   backoff     in (0, 1); growth > 1 (both finite); interval >= 1
 *   stream      cudaStream_t (NULL: the legacy default stream); asynchronous.
 * Returns PSGD_EINVAL, before any launch, for a NULL pointer, a pointer that is not
 * aligned to its element size, or a factor or size out of range. Needs no handle and
 * allocates nothing. */
psgd_status psgd_scale_update(int32_t num_blocks, int32_t num_workers, const int64_t* counts,
                              float* scale, int32_t* streak, double backoff, double growth,
                              int32_t interval, void* stream);

/* Consumer of the decompressed gradient: global-norm clipping and one Adam step with
 * fp32 moments ("Zero-Shot Text-to-Image Generation - 中文验证版" §方法适配: Adam with
 * clipping and a skip rule; "AIGC 基本功|混合精度与数值稳定性" §6.2: the clipping norm is
 * global and taken after unscaling; the update rule is the published bias-corrected
 * Adam). Over every tensor t passed:
 *   n = sqrt(sum_t ||grads[t]||^2); c = min(1, max_norm / n) (c = 1 if max_norm <= 0)
 *   for tensors whose block is not skipped, element-wise with g' = c g:
 *   m <- b1 m + (1 - b1) g'; v <- b2 v + (1 - b2) g'^2;
 *   theta <- theta - lr (m / (1 - b1^step)) / (sqrt(v / (1 - b2^step)) + eps)
 * The norm covers every tensor, skipped or not (psgd_step writes G-hat = 0 for a skipped
 * block). */
#define PSGD_ADAM_MAX_TENSORS 512
typedef struct {
  int32_t num_tensors;              /* T in [1, PSGD_ADAM_MAX_TENSORS] */
  const float* const* grads;        /* [T] host array of device fp32 gradients */
  float* const* params;             /* [T] device fp32 theta, updated */
  float* const* exp_avg;            /* [T] device fp32 m, updated (start at 0) */
  float* const* exp_avg_sq;         /* [T] device fp32 v, updated (start at 0) */
  const int64_t* numel;             /* [T] host element counts (>= 0) */
  const int32_t* block;             /* [T] host resblock index of each tensor (-1: never
                                       skipped), or NULL */
  const uint8_t* skip;              /* device [num_blocks] psgd_step skip flags, or NULL */
  int32_t num_blocks;               /* entries of skip (required with skip) */
  double max_norm;                  /* C; <= 0 disables clipping */
  double lr, beta1, beta2, eps;     /* lr >= 0, 0 <= beta < 1, eps >= 0, all finite */
  int32_t step;                     /* >= 1: the step number after this update */
  float* norm_out;                  /* device fp32 [1]: n before clipping, or NULL */
} psgd_adam_args;

/* Bytes of device workspace psgd_clip_adam needs for these tensor sizes (0 on error). */
size_t psgd_clip_adam_workspace_size(int32_t num_tensors, const int64_t* numel);

/* Enqueue the clip + Adam update on `stream`. workspace: device, 256-byte aligned, at
 * least psgd_clip_adam_workspace_size bytes, caller-owned (its contents are scratch).
 * All device pointers 4-byte aligned. PSGD_EINVAL before any launch on a bad argument.
 * Allocates nothing. */
psgd_status psgd_clip_adam(const psgd_adam_args* args, void* workspace, size_t ws_bytes,
                           void* stream);

/* Uncompressed 32-bit reduction of a gradient that PowerSGD leaves out: the embedding and
 * unembedding (vocabulary x d_model), or any other fp32 tensor outside the compressed
 * matrices ("Zero-Shot Text-to-Image Generation - 中文验证版" §方法适配: embedding,
 * unembedding, gains and biases are reduced in 32-bit, uncompressed; "[논문 정리] Zero-Shot
 * Text-to-Image Generation" §Mixed-Precision Training: Inf/NaN become 0 on unscaling).
 * The arithmetic equals that of psgd_step's gains/biases:
 *   out[i]    = (sum_{w=0..W-1} zero_nonfinite(in[w][i] * (1/scale))) / W   (fp32, in order)
 *   counts[w] = entries of in[w] whose unscaled value is not finite (overwritten)
 * If skip is given and *skip != 0 (e.g. psgd_step's skip flag of a resblock, or a
 * caller's global decision), out is written as 0; the counts are still reported.
 *   num_workers  W in [1, PSGD_UNC_MAX_WORKERS]
 *   in           host array [W] of device fp32 pointers, len entries each, 16-byte aligned
 *   len          entries per worker (>= 0; any value, the tail past a multiple of 4 included)
 *   scale        the tensor's gradient scale s, finite and > 0 (1 when it is not scaled)
 *   out          device fp32 [len], 16-byte aligned; may not overlap an input
 *   counts       device int64 [W], 8-byte aligned
 *   skip         device uint8 [1] or NULL
 * One HBM sweep: W * len * 4 bytes read, len * 4 written. Asynchronous on `stream`;
 * allocates nothing. PSGD_EINVAL before any launch on a bad argument. */
#define PSGD_UNC_MAX_WORKERS 16
psgd_status psgd_reduce_uncompressed(int32_t num_workers, const float* const* in, int64_t len,
                                     float scale, float* out, int64_t* counts,
                                     const uint8_t* skip, void* stream);

/* Wait for `stream`, then report a device-side error raised by an earlier step
 * (PSGD_ETIMEOUT for an expired bounded wait), and clear it. */
psgd_status psgd_check(psgd_handle* h, void* stream);

/* Release the handle's host resources. The workspace stays the caller's. NULL is a no-op. */
psgd_status psgd_finalize(psgd_handle* h);

const char* psgd_strerror(psgd_status s);
const char* psgd_last_error(void);

/* Profiling. psgd_profile_begin creates events for up to `max_steps` later steps. Each of
 * those psgd_step calls records PSGD_NUM_PHASES + 1 events on its stream, at the phase
 * boundaries (ingest | skip and gains/biases | P GEMM | orthonormalisation | Q GEMM |
 * Q reduction | decompress + error update). psgd_profile_end waits for the events. It
 * writes the summed milliseconds of each phase into phase_ms[PSGD_NUM_PHASES] and the
 * number of profiled steps into *steps, then destroys the events. The events are host
 * resources; no device memory is allocated. */
#define PSGD_NUM_PHASES 7
psgd_status psgd_profile_begin(psgd_handle* h, int32_t max_steps);
psgd_status psgd_profile_end(psgd_handle* h, double* phase_ms, int32_t* steps);

/* Total kernel launches this handle has enqueued (all steps so far). */
int64_t psgd_launch_count(psgd_handle* h);

/* Debug: device pointer to M_{b,j,w} (the error-dtype scratch written by the last step),
 * or NULL on a bad index. */
const void* psgd_debug_m(psgd_handle* h, int32_t b, int32_t j, int32_t w);
/* Debug: device pointer to P^_{b,j} of the last step, fp32 m x rp row-major with
 * rp = r rounded up to a multiple of 16 (columns r..rp-1 are 0), or NULL. */
const float* psgd_debug_phat(psgd_handle* h, int32_t b, int32_t j);
/* Debug: after waiting for `stream`, copy the orthonormalisation pass record of matrix
 * (b, j) from the last step into out[PSGD_MAX_ORTH_PASSES * 4]: per pass {final flag,
 * output buffer, shifted flag, dead columns}. Passes after the final one hold stale
 * values. Returns the number of passes that ran (>= 1), or -1 on error. */
#define PSGD_MAX_ORTH_PASSES 4
int32_t psgd_debug_orth(psgd_handle* h, int32_t b, int32_t j, int32_t* out, void* stream);
/* Name of the GEMM engine this handle uses: "tcgen05" or "simt". */
const char* psgd_engine(psgd_handle* h);

/* Orthonormalise one fp32 matrix with scratch that is part of the library image.
 *
 * The pages have no counterpart of this call. It runs the orthonormalisation passes
 * (adaptive shifted CholeskyQR in fp32) that psgd_step applies to each P, for a single
 * matrix, without a handle or a workspace, and it allocates no memory of any kind. It serves callers that hold one P but no
 * handle and cannot allocate at that point: cudaMalloc/cudaFree synchronise the device
 * and would stall the work queued around the call, and a process whose device memory is
 * all handed out to a caching allocator or a fixed budget has none to give.
 *
 *   p     device, fp32, m x r row-major, dense (leading dimension r), 4-byte aligned.
 *         Read only. Entries must be finite.
 *   phat  device, fp32, m x r row-major, dense, 4-byte aligned; receives P^, an
 *         orthonormal basis of span(P) (a numerically dependent column comes out 0).
 *         Must not overlap p. Owned by the caller.
 *   m, r  1 <= r <= m, m <= PSGD_STATIC_MAX_ROWS, r <= PSGD_STATIC_MAX_COLS. Larger
 *         sizes return PSGD_EINVAL (with the limit in psgd_last_error) before any work.
 *   stream  cudaStream_t (NULL: the legacy default stream); the call is asynchronous.
 *
 * Scratch: a fixed __device__ array of 16.1 MiB in each device's copy of the library
 * module (Gram partial sums, R^-1, plan and pass state). The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress, with the device current)
 * and keeps it, with the ID of the context it belongs to; make that first call on each
 * device before any stream capture begins. After a device reset, or when the device's
 * primary context is created anew, the next call is again a first call: it looks the
 * address up again (so it, too, belongs outside a capture).
 * Every call clears the scratch words that must start at zero before it uses them.
 * All calls share the one array: calls that overlap on the GPU (different streams of a
 * device) race on it, so the caller must serialise them, e.g. on one stream.
 * Errors: PSGD_EINVAL for bad arguments, PSGD_ECUDA for a CUDA error (message in
 * psgd_last_error). */
#define PSGD_STATIC_MAX_ROWS 16384
#define PSGD_STATIC_MAX_COLS 128
psgd_status psgd_orthonormalize_static(const float* p, float* phat, int64_t m, int32_t r,
                                       void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PSGD_H_ */
