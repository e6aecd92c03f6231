/*
 * savgb.h - C ABI of the GB300 (sm_103a) chunk-step library.
 *
 * One denoising step of one video chunk of a chunked, flow-matching Diffusion
 * Transformer avatar generator, as described in HeyGen, "Avatar inference at
 * scale":
 *   - section "The underlying model architecture": a DiT trained with flow
 *     matching that attends to rich reference tokens; long videos are made
 *     chunk by chunk, the first chunk relying on the static reference only,
 *     later chunks also on boundary data from the previous chunk;
 *   - section "The streaming framework and pipeline loop": the reference
 *     identity is encoded once per request, then each chunk runs a multi-step
 *     diffusion pass conditioned on the previous chunk's boundary frames;
 *   - section "Constant memory over duration": only the static reference
 *     conditioning and a minimal set of carried tensors live across chunks,
 *     so peak GPU memory does not grow with session length.
 * The pages state the problem, not the operators.  The operator readings
 * this library implements are stated with each call below.
 *
 * Conventions shared by every call
 *   Token tensors are bfloat16, laid out [B][N][H][D] (batch, token, head,
 *   channel), i.e. row-major [B*N][H*D].  Token n of a t x h x w latent block
 *   sits at (t0 + n / (h*w), (n / w) % h, n % w).
 *   Device pointers are caller-owned; the library neither frees them nor keeps
 *   them past the call.  Every device pointer must be 16-byte aligned.
 *   `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *   enqueue work: they return after host-side validation and launch.  Errors
 *   raised by a kernel on the device (a bounded wait that ran out) are
 *   recorded in a per-device error word and reported by savgb_device_check()
 *   or chunk_stream_sync().
 *   Every call returns a savgb_status; on failure savgb_last_error() gives a
 *   thread-local message.  Nothing throws across this boundary.  No call falls
 *   back to the CPU.
 */
#ifndef SAVGB_H
#define SAVGB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility: these declarations are
 * its only exports. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
  SAVGB_OK = 0,
  SAVGB_ERR_INVALID_ARG = -1, /* a size, count or pointer is out of range */
  SAVGB_ERR_UNSUPPORTED = -2, /* valid but not supported (e.g. head_dim not 64/128, no sm_103 device) */
  SAVGB_ERR_ALIGNMENT = -3,   /* a pointer is not 16-byte aligned */
  SAVGB_ERR_OOM = -4,         /* a device allocation failed */
  SAVGB_ERR_CUDA = -5,        /* a CUDA runtime or driver call failed */
  SAVGB_ERR_TIMEOUT = -6,     /* a kernel's bounded wait ran out (device error word) */
  SAVGB_ERR_STATE = -7,       /* call out of order for a stream handle */
} savgb_status;

/* Human-readable name of a status code (static string). */
const char* savgb_status_string(int status);
/* Message of the last failing call on this thread ("" if none). */
const char* savgb_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int savgb_version(void);
/* Kernels this process has enqueued through the library since it was loaded:
 * every launch the CUDA runtime accepted, on any device or stream, counted on
 * the host.  No device work; the difference of two readings counts the
 * launches of the calls between them. */
uint64_t savgb_kernel_launches(void);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns SAVGB_ERR_TIMEOUT (with the kernel and wait that gave up in
 * savgb_last_error()) if a kernel's bounded wait ran out since the last
 * check, SAVGB_ERR_CUDA if the stream reports an error, else SAVGB_OK. */
int savgb_device_check(void* stream);

/* Diagnostic with no counterpart on the pages: launches one block that waits,
 * through the same bounded wait the library's kernels use, on a barrier that
 * nothing arrives on, for at most limit_ns nanoseconds (0 < limit_ns <= 1e10).
 * A following savgb_device_check() then returns SAVGB_ERR_TIMEOUT.  It checks
 * failure reporting without faulting or hanging the GPU. */
int savgb_watchdog_selftest(uint64_t limit_ns, void* stream);

/* Diagnostic with no counterpart on the pages: arms a one-shot fault in the
 * next launch of one of the library's kernels, so that a test can run that
 * kernel's own give-up path without faulting or hanging the GPU.
 *   SAVGB_FAULT_ATTENTION_K_TILE  the attention kernel (any of its entry
 *       points, the chunk-stream steps included): in the block of batch 0,
 *       head 0, first query block, the key producer skips the copy of key
 *       tile `index` (and the arrival that goes with it);
 *   SAVGB_FAULT_WO_PAIR_RELAY  the W_o CTA-pair kernel (out_proj_euler_step
 *       with no v_out and hid_out % 256 == 0, and the stream steps): the odd
 *       CTA of the first cluster skips its "stage full" relay of k-block
 *       iteration `index`.  Other W_o launches leave the arm in place.
 * Every bounded wait of that launch gives up after limit_ns nanoseconds
 * (0 < limit_ns <= 1e10) instead of 2 s; the kernel records the timeout in
 * the device error word, waits (bounded) for its own copies and MMAs in
 * flight, frees its tensor memory and returns, and the next
 * savgb_device_check() returns SAVGB_ERR_TIMEOUT.  That launch's outputs are
 * undefined.  The arm is process-wide and taken by the next launch of that
 * kernel from any thread; index < 0 disarms.  SAVGB_ERR_INVALID_ARG for an
 * unknown kind or a limit out of range. */
#define SAVGB_FAULT_ATTENTION_K_TILE 1
#define SAVGB_FAULT_WO_PAIR_RELAY 2
int savgb_arm_wait_fault(int kind, int index, uint64_t limit_ns);

/* --------------------------------------------------------------------------
 * rope3d_apply - 3D (t, h, w) rotary position embedding.
 *
 * Positions of the latent tokens in time and space (the chunked latent video
 * of "The underlying model architecture").  Reading: the D/2 channel pairs are
 * split [t | h | w]; each spatial axis owns floor(D/6) pairs and time the rest
 * (D=128: 22/21/21, D=64: 12/10/10).  Pair j of an axis with P pairs turns at
 * omega_j = base^(-j/P) radians per position; the adjacent pair (a, b) becomes
 * (a cos th - b sin th, a sin th + b cos th), th = pos * omega_j.
 *
 *   in, out   bf16 [B][n_tokens][H][D]; in == out is allowed (in place).
 *   n_tokens  must equal grid_t * grid_h * grid_w (>= 1).
 *   D         even, 8 <= D <= 256, D % 8 == 0.
 *   t0        time of the first frame (chunk tokens 0, boundary -T_b, ...).
 *   base      rotary base (> 0), typically 10000.
 * Math in fp32 from the bf16 inputs; output rounded to bf16 (nearest even).
 * Limits: grid_h, grid_w <= 4096, grid_t <= 4096 and the three angle tables
 * (grid_t*P_t + grid_h*P_h + grid_w*P_w entries) fit 96 KiB of shared memory.
 * ------------------------------------------------------------------------ */
int rope3d_apply(const void* in, void* out, int B, int64_t n_tokens, int H, int D, int grid_t,
                 int grid_h, int grid_w, int t0, double base, void* stream);

/* One key/value segment: bf16 k and v, each [B][n_tokens][H][D] with the
 * same B, H, D as the queries.  n_tokens may be 0 (then k and v are unused). */
typedef struct {
  const void* k;
  const void* v;
  int64_t n_tokens;
} savgb_kv_segment;
/* The same segment under the name the problem statement's interface uses. */
typedef savgb_kv_segment kv_segment_t;

/* --------------------------------------------------------------------------
 * chunk_attention - queries of the current chunk attend over the
 * concatenation of up to three key/value segments, in practice
 * [static reference | previous chunk's boundary | current chunk]
 * ("The underlying model architecture": rich reference tokens and boundary
 * data from previous segments; "The streaming framework and pipeline loop":
 * the chunk is conditioned on the previous chunk's boundary frames).
 *
 * Reading: no mask; O = softmax(Q K^T * scale) V per (batch, head).
 *   q        bf16 [B][n_q][H][D], already rotated.
 *   segs     n_segs (1..3) segments; their total token count must be >= 1.
 *   scale    softmax scale; <= 0 selects 1/sqrt(D).
 *   o        bf16 [B][n_q][H][D] output (must not alias q or any k/v).
 *   lse      optional fp32 [B][H][n_q]: natural-log sum of exp(scale*q.k).
 * D must be 64 or 128.  bf16 tensor-core products, fp32 accumulation; the
 * probabilities are bf16 (the PV operand), from one packed bf16 exp2 per two
 * scores with their exponents rounded to bf16, and the row sums add those
 * bf16 values in fp32.  With lse non-NULL the kernel instead takes fp32
 * exponentials and exact fp32 row sums (the packed form's sums run ~0.3 %
 * low, which cancels in O but not in lse); that form is a few percent slower.
 * It also serves every scale above 1.25 x 1/sqrt(D): the packed form rounds
 * each exponent to bf16, whose error grows with the spread of the logits.
 * Against an fp64 reference, on unit-variance q and k at the default scale
 * both forms stay near 2.5e-3 max-abs; for logits 2x to 6x sharper the fp32
 * form stays below 1.7e-2 while the packed one can pass 2e-2.  Callers whose
 * logits are sharper than that through their data rather than the scale can
 * ask for the fp32 form with exact_softmax in a chunk stream's config.
 * ------------------------------------------------------------------------ */
int chunk_attention(const void* q, int B, int64_t n_q, int H, int D, const savgb_kv_segment* segs,
                    int n_segs, float scale, void* o, float* lse, void* stream);

/* chunk_attention_qrope - chunk_attention with the 3D RoPE of the queries
 * applied inside the kernel: q holds the chunk's queries BEFORE rotation,
 * laid out as a grid_t x grid_h x grid_w token grid starting at time t0 (the
 * rope3d_apply reading: D/2 pairs split [t | h | w], pair j of an axis with P
 * pairs turning at base^(-j/P)).  Each block rotates its query tiles in
 * shared memory after loading them, which removes one read and one write of
 * q from HBM.  The cos/sin table ([t rows | h | w] x pairs, fp32) is built on
 * `stream` by a small kernel into a stream-ordered temporary
 * (cudaMallocAsync / cudaFreeAsync, a few KB to tens of KB) and copied into
 * each block's shared memory; chunk streams build theirs once at create, and
 * chunk_attention_qrope_with_table (below) takes one the caller built.
 * Keys must already be rotated.  Other arguments and errors as
 * chunk_attention; n_q must equal grid_t*grid_h*grid_w.
 * SAVGB_ERR_UNSUPPORTED when a block's part of the table, 8 * (r*Pt +
 * grid_h*Ph + grid_w*Pw) bytes with (Pt, Ph, Pw) the pairs per axis and r <=
 * 255/(grid_h*grid_w) + 2 the time rows one 256-query block spans, exceeds
 * the shared memory left beside the operands: 34560 bytes at D = 128 (a
 * grid_h + grid_w of about 200), 67328 at D = 64.
 * ("The underlying model architecture": chunked latent video, reference and
 * boundary tokens as context.) */
int chunk_attention_qrope(const void* q, int B, int64_t n_q, int H, int D, int grid_t, int grid_h,
                          int grid_w, int t0, double base, const savgb_kv_segment* segs, int n_segs,
                          float scale, void* o, float* lse, void* stream);

/* chunk_attention_qrope with a caller-built cos/sin table, for callers that
 * run the stand-alone fused call in a loop and want no allocation per call.
 *   chunk_attention_qrope_table_bytes: host query, *bytes = the table's size
 *     for a grid_t x grid_h x grid_w query grid at head_dim D (64 or 128;
 *     grid sizes in [1, 4096]).  No device work.
 *   chunk_attention_qrope_build_table: fills `table` (caller-owned device
 *     memory of at least that many bytes, 16-byte aligned) on `stream` for
 *     time values t0 .. t0+grid_t-1 and the whole grid_h x grid_w grid at
 *     rotary base `base` (one small kernel).
 *   chunk_attention_qrope_with_table: chunk_attention_qrope that reads such a
 *     table instead of building one; D, the grid and t0 must be those the
 *     table was built for (the table carries the base).  The table must stay
 *     unchanged until the call's kernel has run (stream order).  Other
 *     arguments, errors and limits as chunk_attention_qrope.
 * (Library facilities over the same computation; the pages have no
 * counterpart.) */
int chunk_attention_qrope_table_bytes(int D, int grid_t, int grid_h, int grid_w, int64_t* bytes);
int chunk_attention_qrope_build_table(void* table, int D, int grid_t, int grid_h, int grid_w, int t0, double base,
                                      void* stream);
int chunk_attention_qrope_with_table(const void* q, int B, int64_t n_q, int H, int D, int grid_t, int grid_h,
                                     int grid_w, int t0, const void* table, const savgb_kv_segment* segs,
                                     int n_segs, float scale, void* o, float* lse, void* stream);

/* chunk_attention_qrope_fits - host query, no device work: *fits = 1 when
 * the block's part of the cos/sin table for a grid_t x grid_h x grid_w query
 * grid fits in the attention kernel's shared memory (the limit stated for
 * chunk_attention_qrope), else 0; *fits = 0 for a head_dim other than 64 or
 * 128.  The same test picks the RoPE form of chunk_stream_step and
 * chunk_step_noalloc: q rotated inside the attention kernel when it fits,
 * one RoPE pass over q and k otherwise.  SAVGB_ERR_INVALID_ARG for a grid
 * size below 1 or a NULL fits.  (A library facility; the pages have no
 * counterpart.) */
int chunk_attention_qrope_fits(int D, int grid_t, int grid_h, int grid_w, int* fits);

/* --------------------------------------------------------------------------
 * out_proj_euler_step - output projection of the attention, taken as the
 * flow-matching velocity, followed by one explicit Euler step of the flow
 * ("The underlying model architecture": a DiT trained with flow matching;
 * "The streaming framework and pipeline loop": a multi-step diffusion pass).
 *
 *   v = O W_o^T (+ bias);  x <- x + dt * v
 *   o      bf16 [M][hid_in] (the attention output, rows = B*n_q tokens).
 *   w_o    bf16 [hid_out][hid_in] (PyTorch Linear layout).
 *   bias   optional fp32 [hid_out].
 *   x      fp32 [M][hid_out], updated in place.
 *   v_out  optional fp32 [M][hid_out]: receives v (for inspection).
 * hid_in % 8 == 0, hid_out % 16 == 0.  bf16 tensor-core product, fp32
 * accumulation; the update is fused into the GEMM epilogue.
 * ------------------------------------------------------------------------ */
int out_proj_euler_step(const void* o, const void* w_o, const float* bias, float* x, int64_t M,
                        int hid_in, int hid_out, float dt, float* v_out, void* stream);

/* --------------------------------------------------------------------------
 * qkv_rope_project - QKV projection of one DiT attention block with the 3D
 * RoPE of q and k fused into the GEMM epilogue ("The underlying model
 * architecture": the denoiser is a Diffusion Transformer; a single attention
 * block with stand-in weights takes the place of the network here).
 *   [q | k | v] = x W_qkv^T;  q, k rotated at (t0 + n/(h*w), (n/w)%h, n%w)
 *   x       bf16 [B][n_tokens][H*D]   (n_tokens = grid_t*grid_h*grid_w)
 *   w_qkv   bf16 [3*H*D][H*D] = [W_q; W_k; W_v] (PyTorch Linear layout)
 *   q, k, v bf16 [B][n_tokens][H][D] outputs.
 * D must be 64 or 128; bf16 tensor-core product, fp32 accumulation, rotation
 * in fp32, outputs rounded to bf16.
 * ------------------------------------------------------------------------ */
int qkv_rope_project(const void* x_bf16, const void* w_qkv, void* q, void* k, void* v, int B,
                     int64_t n_tokens, int H, int D, int grid_t, int grid_h, int grid_w, int t0,
                     double base, void* stream);

/* --------------------------------------------------------------------------
 * flow_time_grid - step sizes of the sampling grid (host only).
 * Reading of "multi-step diffusion pass": noise levels sigma_i = 1 - i/steps,
 * warped by sigma' = shift*sigma / (1 + (shift-1)*sigma), dt_i = sigma'_i -
 * sigma'_{i+1} > 0, sum 1.  shift = 1 is the uniform grid.
 *   dt_out  host array of `steps` doubles.
 * ------------------------------------------------------------------------ */
int flow_time_grid(int steps, double shift, double* dt_out);

/* --------------------------------------------------------------------------
 * Chunk stream: the rolling state of one or more sessions.
 * ("The underlying model architecture": the first chunk relies on the static
 * reference alone, later chunks also on boundary data; "The streaming
 * framework and pipeline loop": the reference is encoded once per request;
 * "Constant memory over duration": only the reference conditioning and a
 * minimal carried state survive a chunk, so memory is fixed by the chunk
 * size, not by the session length.)
 *
 * The handle owns one device arena, sized at create and never grown: the
 * rotated reference K and V, two boundary slots (in use / being captured) and
 * the per-step scratch for rotated Q, rotated K and the attention output.
 * Boundary reading: the pre-RoPE K and V of the last `boundary_frames`
 * frames of a chunk, taken at its last denoising step, with K rotated to
 * t = -boundary_frames .. -1 of the next chunk's local time.  Chunk-local time
 * keeps every angle bounded however long the session runs.
 * A handle is not thread-safe; separate handles are independent.
 * ------------------------------------------------------------------------ */
typedef struct {
  int B;               /* sessions batched in one launch (independent) */
  int H, D;            /* heads, head_dim (64 or 128) */
  int F;               /* latent frames per chunk */
  int grid_h, grid_w;  /* latent tokens per frame = grid_h * grid_w */
  int ref_frames;      /* reference frames (>= 1), at t = ref_t-ref_frames+1 .. ref_t */
  int boundary_frames; /* frames carried to the next chunk, 0 <= boundary_frames <= F */
  int ref_t;           /* time of the last reference frame, e.g. -1 */
  double rope_base;    /* rotary base, e.g. 10000 */
  float softmax_scale; /* <= 0 selects 1/sqrt(D) */
  int interp_chunks;   /* nonzero: keep the anchors of interpolation chunks (needs F >= 3) */
  int qkv_block;       /* nonzero: reserve room for chunk_stream_block_step */
  int host_io;         /* 0, or the device input slots of chunk_stream_step_host: 2 to 8 (1 means 2) */
  int exact_softmax;   /* nonzero: the steps' attention takes fp32 exponentials (see chunk_attention) */
} chunk_stream_config;
/* The same config under the name the problem statement's interface uses. */
typedef chunk_stream_config chunk_stream_config_t;

typedef struct chunk_stream chunk_stream_t;

/* Validates the config, allocates the arena on the current device and binds
 * the handle to `stream` (cudaStream_t).  *out receives the handle. */
int chunk_stream_create(const chunk_stream_config* cfg, void* stream, chunk_stream_t** out);

/* Copies the reference K (rotated once, here) and V, bf16 [B][R][H][D] with
 * R = ref_frames*grid_h*grid_w, into the arena.  Call once before the first
 * step; calling again replaces the reference and restarts the stream. */
int chunk_stream_set_reference(chunk_stream_t* s, const void* k_ref, const void* v_ref);

/* One denoising step of the current chunk:
 *   rope3d(q), rope3d(k) at chunk-local positions -> chunk_attention over
 *   [reference | boundary | chunk] -> out_proj_euler_step(x, dt).
 *   q, k, v  bf16 [B][N][H][D], N = F*grid_h*grid_w (pre-RoPE, caller-owned).
 *   w_o      bf16 [H*D][H*D]; bias optional fp32 [H*D].
 *   x        fp32 [B*N][H*D], updated in place.
 * With is_last_step != 0 the boundary for the next chunk is captured from
 * this step's k and v. */
int chunk_stream_step(chunk_stream_t* s, const void* q, const void* k, const void* v,
                      const void* w_o, const float* bias, float* x, float dt, int is_last_step);

/* chunk_stream_step with the step's inputs in HOST memory and, optionally,
 * the updated state read back to host memory: the whole step through one
 * call, host to host, as a serving loop that receives each step's q, k, v
 * from the host and hands the state back would run it.  Needs host_io in the
 * config: the arena then holds host_io (at least 2, at most 8) device input
 * slots of 3 x B*N*H*D bf16 and two staging copies of the state, B*N*H*D fp32
 * each; more slots let the uploads run further ahead of the compute and ride
 * out a slow spell of the host link.
 *   q_host, k_host, v_host  bf16 [B][N][H][D] in host memory; page-locked
 *       (cudaHostAlloc / cudaHostRegister) for the upload to overlap compute,
 *       pageable memory also works but its copy blocks the calling thread.
 *   x       fp32 [B*N][H*D] DEVICE state, updated in place (it stays resident).
 *   x_host  optional fp32 [B*N][H*D] host buffer (page-locked to overlap):
 *       receives x after this step.
 * The call enqueues and returns.  The upload goes into input slot (call
 * count mod slots) on an internal copy stream once the step that last used
 * that slot has finished with it; the step runs on the handle's stream once its
 * upload has landed.  With x_host, the step's W_o update also writes the new x
 * into one of the two staging copies (alternately), and the read-back reads
 * that copy on a second internal copy stream after the step; only the W_o
 * update that writes the same copy again, two such calls later, waits for it.
 * So consecutive calls overlap the upload of step i+1 and the read-back of
 * step i with the compute of step i+1, and a read-back has two steps' time to
 * land before it holds anything up.
 * Host buffers passed to a call must stay valid and unchanged (inputs) or
 * unread (x_host) until chunk_stream_sync() returns, or until the handle's
 * stream has passed a chunk_stream_join_copies() enqueued after the call.
 * SAVGB_ERR_STATE without host_io.  Otherwise as chunk_stream_step. */
int chunk_stream_step_host(chunk_stream_t* s, const void* q_host, const void* k_host, const void* v_host,
                           const void* w_o, const float* bias, float* x, float dt, int is_last_step,
                           float* x_host);
/* Makes the handle's stream wait for every upload and read-back that
 * chunk_stream_step_host has enqueued so far (work enqueued on the stream
 * afterwards, an event for one, comes after them).  Returns at once. */
int chunk_stream_join_copies(chunk_stream_t* s);

/* --------------------------------------------------------------------------
 * Interpolation (I) chunks ("Boundary continuity and chunk consistency"):
 * N chunks form the primary timeline and I chunks smooth the transitions
 * between consecutive N chunks, in the order N0, N1, I0, N2, I1, N3, I2, ...
 * I_k runs after N_k and N_{k+1} are finished.  Reading: an I chunk spans F
 * latent frames whose first and last frames are anchors - the last frame of
 * N_k (at t = 0) and the first frame of N_{k+1} (at t = F-1), both the
 * pre-RoPE K and V of their chunk's final step - and whose F-2 interior
 * frames are generated; anchor predictions are discarded, so only interior
 * frames are queries.  Keys/values: [reference | anchors | interior].
 * With interp_chunks set, the last step of every N chunk keeps its first and
 * last frame in two fixed anchor slots.
 *
 * chunk_stream_istep: one denoising step of the pending I chunk I_k,
 *   k = chunk_stream_ichunk_index().  q, k, v: bf16 [B][(F-2)*h*w][H][D]
 *   interior tokens (before RoPE, chunk-local t = 1..F-2); x fp32
 *   [B*(F-2)*h*w][H*D].  Needs N_k and N_{k+1} finished: SAVGB_ERR_STATE
 *   otherwise.  If N_{k+2} has also finished, the anchors of I_k are gone and
 *   the pending I chunk moves on to I_{done-2} (I chunks not run are skipped).
 * chunk_stream_end_ichunk: the pending I chunk is done; the next one is pending.
 * ------------------------------------------------------------------------ */
int chunk_stream_istep(chunk_stream_t* s, const void* q, const void* k, const void* v,
                       const void* w_o, const float* bias, float* x, float dt);
int chunk_stream_end_ichunk(chunk_stream_t* s);
/* Index of the pending I chunk (0 before the first). */
int chunk_stream_ichunk_index(const chunk_stream_t* s, int64_t* index);

/* One denoising step of the current chunk through one DiT attention block:
 * the state itself is projected, x -> bf16 -> qkv_rope_project (q, k
 * rotated) -> chunk_attention over [reference | boundary | chunk] ->
 * out_proj_euler_step(x, dt).  Needs qkv_block in the config.
 *   w_qkv bf16 [3*H*D][H*D]; w_o bf16 [H*D][H*D]; bias optional fp32 [H*D];
 *   x fp32 [B*N][H*D], updated in place.
 * With is_last_step the next chunk's boundary is taken from this step's
 * projected k (before RoPE) and v.  Block steps keep no I-chunk anchors. */
int chunk_stream_block_step(chunk_stream_t* s, const void* w_qkv, const void* w_o, const float* bias,
                            float* x, float dt, int is_last_step);

/* Ends the current chunk: the boundary captured at its last step becomes the
 * boundary of the next chunk, and the chunk index advances.  Returns
 * SAVGB_ERR_STATE if no step of the chunk had is_last_step set (with
 * boundary_frames > 0). */
int chunk_stream_end_chunk(chunk_stream_t* s);

/* Optional timing of the next step: `events` holds 4 cudaEvent_t that the
 * next chunk_stream_step records on the handle's stream at its start, after
 * the RoPE launch, after the attention launch and after the W_o/Euler launch.
 * They apply to one step only; NULL clears them.  (A library facility with
 * no counterpart on the pages: it lets a caller attribute step time to the
 * kernels as they run inside a loop.) */
int chunk_stream_set_step_events(chunk_stream_t* s, void* const* events);

/* Synchronises the handle's stream (and, with host_io, its copy streams) and
 * reports device-side errors. */
int chunk_stream_sync(chunk_stream_t* s);

/* Read-only view of the state: chunk index, boundary tokens in use (0 on
 * chunk 0), bytes of the device arena, and device pointers to the boundary K
 * (rotated) and V in use (NULL when there is no boundary). */
int chunk_stream_info(const chunk_stream_t* s, int64_t* chunk_index, int64_t* boundary_tokens,
                      int64_t* arena_bytes, const void** boundary_k, const void** boundary_v);

/* *fused = 1 when the steps of this stream rotate q inside the attention
 * kernel (chunk_attention_qrope with a cos/sin table built once at create and
 * kept in the arena; the RoPE pass then rotates k only), 0 when one pass
 * rotates q and k before chunk_attention.  The fused form is used whenever its
 * table fits in the kernel's shared memory; both give the same results to
 * bf16 rounding. */
int chunk_stream_fused_q_rope(const chunk_stream_t* s, int* fused);

/* Checkpoint of the rolling state (chunk index, boundary K/V in use, and with
 * interp_chunks the I-chunk index and both anchor slots) into a host buffer.  With buf == NULL only *size_out is set.  Synchronises the
 * stream.  The reference is not part of the state (it is set again on
 * resume). */
int chunk_stream_export_state(chunk_stream_t* s, void* buf, size_t cap, size_t* size_out);
/* Restores a state written by chunk_stream_export_state of a handle with the
 * same config.  SAVGB_ERR_INVALID_ARG on a size or config mismatch. */
int chunk_stream_import_state(chunk_stream_t* s, const void* buf, size_t size);

/* Frees the arena and the handle (after synchronising its stream). */
int chunk_stream_destroy(chunk_stream_t* s);

/* --------------------------------------------------------------------------
 * chunk_step_noalloc - one chunk denoising step that allocates no device
 * memory.  The pages have no counterpart to this call: it serves callers that
 * cannot call cudaMalloc, such as a plugin inside a serving runtime that owns
 * every device allocation and offers plugins no allocator, or a real-time loop
 * that may not allocate (or synchronise the device through an allocation) once
 * the session runs.  Such callers cannot create a chunk_stream handle.
 *
 * Computes what chunk_stream_step computes: RoPE of q and k at chunk-local
 * positions, attention over [context segments | chunk], and the W_o GEMM with
 * the Euler update x <- x + dt * (O W_o^T + bias).  The caller keeps the
 * rolling state itself: `context` holds 0 to 2 already-rotated segments (the
 * reference, then the boundary, as rope3d_apply produces them), each bf16
 * [B][n][H][D].  q, k, v: bf16 [B][N][H][D], N = F*grid_h*grid_w; w_o bf16
 * [H*D][H*D]; bias optional fp32 [H*D]; x fp32 [B*N][H*D], updated in place.
 *
 * Like the stream, the step rotates q inside the attention kernel when that
 * kernel's cos/sin table fits in its shared memory (rebuilt by every call),
 * else q and k in one RoPE pass.  Its intermediates (rotated k, the attention
 * output: 2 x B*N*H*D bf16, plus the table or rotated q, each rounded up to
 * 256 bytes) live in one file-scope device array of
 * SAVGB_NOALLOC_SCRATCH_BYTES, which every device that loads the
 * library holds until the process exits.  Larger steps are rejected with
 * SAVGB_ERR_INVALID_ARG.  The array's address is looked up on the first call
 * made on each device; make that call before any stream capture.  All calls
 * share the array, so calls that overlap on the GPU race; nothing in it needs
 * clearing between calls.
 * ------------------------------------------------------------------------ */
#define SAVGB_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int chunk_step_noalloc(const void* q, const void* k, const void* v, const savgb_kv_segment* context,
                       int n_context, const void* w_o, const float* bias, float* x, float dt, int B,
                       int H, int D, int F, int grid_h, int grid_w, double rope_base,
                       float softmax_scale, void* stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* SAVGB_H */
