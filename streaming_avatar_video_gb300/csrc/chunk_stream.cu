// Chunk stream: the rolling state of B independent sessions.
//
// HeyGen, "Avatar inference at scale":
//   - "The underlying model architecture": the first chunk relies on the
//     static reference only; later chunks also use boundary data from the
//     previous chunk.
//   - "The streaming framework and pipeline loop": the reference identity is
//     encoded once per request; each chunk runs a multi-step diffusion pass
//     conditioned on the previous chunk's boundary frames.
//   - "Constant memory over duration": only the reference conditioning and a
//     minimal carried state survive a chunk; peak memory is set by the chunk
//     size, not by the session length.
//
// The handle owns one device arena allocated at create and never grown:
//   ref_k (rotated once) | ref_v | boundary k/v x 2 slots | q_rot | k_rot | o
//   | (interpolation anchors, block-step v) | cos/sin table of the q RoPE
// A step enqueues, on the handle's stream: RoPE of k, attention over
// [reference | boundary | chunk] with the RoPE of q applied inside the kernel
// from the table built at create (or, when that table does not fit in the
// kernel's shared memory, RoPE of q and k in one launch and the plain
// attention), then the W_o GEMM with the Euler update fused into its
// epilogue.  The last step of a chunk also rotates
// the tail frames of its k into the spare boundary slot (t = -T_b .. -1) and
// copies the tail of v; end_chunk swaps the slots.
#include <cuda_bf16.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <new>

#include "common.h"

using namespace savgb;

// input slots of chunk_stream_step_host: host_io in the config (1 means 2)
constexpr int kMaxInSlots = 8;

struct chunk_stream {
  chunk_stream_config cfg;
  cudaStream_t stream;
  int device;
  int64_t n_tok;     // tokens per chunk
  int64_t n_ref;     // reference tokens
  int64_t n_bnd;     // boundary tokens once a boundary exists
  int64_t hid;
  void* arena;
  int64_t arena_bytes;
  __nv_bfloat16_raw* ref_k;
  __nv_bfloat16_raw* ref_v;
  __nv_bfloat16_raw* bnd_k[2];
  __nv_bfloat16_raw* bnd_v[2];
  __nv_bfloat16_raw* q_rot;
  __nv_bfloat16_raw* k_rot;
  __nv_bfloat16_raw* o;
  // interpolation chunks: slot k%2 holds the anchors of I_k, [B][2 frames][H][D]:
  // N_k's last frame rotated to t = 0, then N_{k+1}'s first frame rotated to t = F-1
  __nv_bfloat16_raw* anc_k[2];
  __nv_bfloat16_raw* anc_v[2];
  __nv_bfloat16_raw* v_buf;  // projected v of a block step (qkv_block); its bf16 x shares `o`
  // the RoPE of q runs inside the attention kernel when its cos/sin table (t
  // in [0, F) and the whole grid, built once here) fits in shared memory
  bool qrope;
  void* qrope_tab;
  int64_t ichunk_index;
  int cur;             // boundary slot in use
  int64_t bnd_in_use;  // 0 on chunk 0
  bool captured;
  bool ref_set;
  int64_t chunk_index;
  cudaEvent_t step_events[4];  // recorded by the next step, then cleared
  bool have_events;
  // host_io: n_slots device input slots [q | k | v] filled from host memory
  // on copy_in; the state read back on copy_out from one of two staging
  // copies that the W_o update writes beside x (chunk_stream_step_host)
  int n_slots;
  __nv_bfloat16_raw* in_slot[kMaxInSlots][3];
  float* x_stage[2];
  cudaStream_t copy_in, copy_out;
  cudaEvent_t ev_loaded[kMaxInSlots], ev_freed[kMaxInSlots], ev_step_done, ev_out_done;
  cudaEvent_t ev_stage_read[2];  // the read-back from that staging copy has landed
  bool slot_used[kMaxInSlots];
  int next_slot;
  bool stage_pending[2];  // a read-back from that staging copy is in flight
  int next_stage;
  bool out_pending;  // some read-back is in flight (ev_out_done: the latest)
  bool host_used;    // copies were enqueued since the last join / sync
};

namespace {

constexpr uint64_t kStateMagic = 0x5341564742535431ull;  // "SAVGBST1"

struct StateHeader {
  uint64_t magic;
  int32_t B, H, D, F, grid_h, grid_w, boundary_frames, interp;
  int64_t chunk_index;
  int64_t bnd_in_use;
  int64_t payload_bytes;
  int64_t ichunk_index;
  int64_t reserved;
};

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

int validate_config(const chunk_stream_config* c) {
  if (!c) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: null config");
  if (c->B < 1 || c->H < 1 || c->F < 1 || c->grid_h < 1 || c->grid_w < 1)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: B, H, F, grid_h, grid_w must be >= 1");
  if (c->D != 64 && c->D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_stream: head_dim %d (64 or 128 supported)", c->D);
  if (c->ref_frames < 1) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: ref_frames must be >= 1");
  if (c->boundary_frames < 0 || c->boundary_frames > c->F)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: boundary_frames must be in [0, F]");
  if (!(c->rope_base > 0.0) || !std::isfinite(c->rope_base))
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: rope_base must be finite and > 0");
  const int64_t hid = (int64_t)c->H * c->D;
  if (hid % 16) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: H*D must be a multiple of 16");
  if (c->interp_chunks && c->F < 3)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: interpolation chunks need F >= 3");
  if (c->host_io < 0 || c->host_io > kMaxInSlots)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream: host_io must be 0 (off) or 1 to %d input slots (1 means 2)",
                kMaxInSlots);
  return SAVGB_OK;
}

// Copy streams and events of chunk_stream_step_host.
int host_io_init(chunk_stream* s) {
  SAVGB_CUDA(cudaStreamCreateWithFlags(&s->copy_in, cudaStreamNonBlocking));
  SAVGB_CUDA(cudaStreamCreateWithFlags(&s->copy_out, cudaStreamNonBlocking));
  for (int i = 0; i < s->n_slots; ++i) {
    SAVGB_CUDA(cudaEventCreateWithFlags(&s->ev_loaded[i], cudaEventDisableTiming));
    SAVGB_CUDA(cudaEventCreateWithFlags(&s->ev_freed[i], cudaEventDisableTiming));
    s->slot_used[i] = false;
  }
  SAVGB_CUDA(cudaEventCreateWithFlags(&s->ev_step_done, cudaEventDisableTiming));
  SAVGB_CUDA(cudaEventCreateWithFlags(&s->ev_out_done, cudaEventDisableTiming));
  for (int i = 0; i < 2; ++i) {
    SAVGB_CUDA(cudaEventCreateWithFlags(&s->ev_stage_read[i], cudaEventDisableTiming));
    s->stage_pending[i] = false;
  }
  s->next_slot = 0;
  s->next_stage = 0;
  s->out_pending = false;
  s->host_used = false;
  return SAVGB_OK;
}

void host_io_release(chunk_stream* s) {
  if (s->copy_in) cudaStreamSynchronize(s->copy_in);
  if (s->copy_out) cudaStreamSynchronize(s->copy_out);
  for (int i = 0; i < kMaxInSlots; ++i) {
    if (s->ev_loaded[i]) cudaEventDestroy(s->ev_loaded[i]);
    if (s->ev_freed[i]) cudaEventDestroy(s->ev_freed[i]);
  }
  if (s->ev_step_done) cudaEventDestroy(s->ev_step_done);
  if (s->ev_out_done) cudaEventDestroy(s->ev_out_done);
  for (int i = 0; i < 2; ++i)
    if (s->ev_stage_read[i]) cudaEventDestroy(s->ev_stage_read[i]);
  if (s->copy_in) cudaStreamDestroy(s->copy_in);
  if (s->copy_out) cudaStreamDestroy(s->copy_out);
}

// The staging copy of x that a host step's W_o update writes: the read-back
// from it two host steps back must have landed first.  nullptr for stage < 0.
int take_stage(chunk_stream* s, int stage, float** x_copy) {
  *x_copy = nullptr;
  if (stage < 0) return SAVGB_OK;
  if (s->stage_pending[stage]) SAVGB_CUDA(cudaStreamWaitEvent(s->stream, s->ev_stage_read[stage], 0));
  s->stage_pending[stage] = false;
  *x_copy = s->x_stage[stage];
  return SAVGB_OK;
}

RopeArgs rope_args(const chunk_stream* s, const void* in, void* out, int64_t in_bs, int64_t out_bs,
                   int grid_t, int t0) {
  const chunk_stream_config& c = s->cfg;
  return RopeArgs{in, out, c.B, (int64_t)grid_t * c.grid_h * c.grid_w, c.H, c.D, grid_t,
                  c.grid_h, c.grid_w, t0, c.rope_base, in_bs, out_bs};
}

}  // namespace

extern "C" {

int chunk_stream_create(const chunk_stream_config* cfg, void* stream, chunk_stream_t** out) {
  savgb::ApiRange api_range_("savgb:chunk_stream_create");
  clear_error();
  if (!out) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_create: null out");
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  if ((rc = check_device(nullptr))) return rc;
  chunk_stream* s = new (std::nothrow) chunk_stream();
  if (!s) return fail(SAVGB_ERR_OOM, "chunk_stream_create: host allocation");
  s->cfg = *cfg;
  s->stream = static_cast<cudaStream_t>(stream);
  cudaGetDevice(&s->device);
  const chunk_stream_config& c = *cfg;
  s->hid = (int64_t)c.H * c.D;
  const int64_t fr = (int64_t)c.grid_h * c.grid_w;
  s->n_tok = c.F * fr;
  s->n_ref = c.ref_frames * fr;
  s->n_bnd = c.boundary_frames * fr;
  // validate every launch shape once, up front
  RopeArgs probe = rope_args(s, (void*)16, (void*)16, 0, 0, c.F, 0);
  if ((rc = validate_rope(probe))) { delete s; return rc; }
  probe = rope_args(s, (void*)16, (void*)16, 0, 0, c.ref_frames, c.ref_t - c.ref_frames + 1);
  if ((rc = validate_rope(probe))) { delete s; return rc; }
  const int64_t tok_bytes = s->hid * 2 * c.B;  // one token of all sessions
  const int64_t ref_b = round_up(s->n_ref * tok_bytes, 256);
  const int64_t bnd_b = round_up((s->n_bnd > 0 ? s->n_bnd : 1) * tok_bytes, 256);
  const int64_t tok_b = round_up(s->n_tok * tok_bytes, 256);
  const int64_t anc_b = c.interp_chunks ? round_up(2 * fr * tok_bytes, 256) : 0;
  const int64_t vbuf_b = c.qkv_block ? tok_b : 0;
  s->qrope = qrope_fits(c.D, c.F, c.grid_h, c.grid_w);
  const int64_t tab_b = s->qrope ? round_up(rope_q_table_bytes(c.D, c.F, c.grid_h, c.grid_w), 256) : 0;
  s->n_slots = c.host_io ? (c.host_io < 2 ? 2 : c.host_io) : 0;
  const int64_t in_b = 3 * s->n_slots * tok_b;
  const int64_t stage_b = c.host_io ? round_up(s->n_tok * s->hid * 4 * c.B, 256) : 0;  // fp32 copies of x
  s->arena_bytes = 2 * ref_b + 4 * bnd_b + 3 * tok_b + 4 * anc_b + vbuf_b + tab_b + in_b + 2 * stage_b;
  const char* cap = getenv("SAVGB_ARENA_LIMIT_BYTES");
  if (cap && *cap) {
    const long long lim = atoll(cap);
    if (lim >= 0 && s->arena_bytes > lim) {
      const long long need = (long long)s->arena_bytes;
      delete s;
      return fail(SAVGB_ERR_OOM, "chunk_stream_create: arena of %lld bytes exceeds SAVGB_ARENA_LIMIT_BYTES=%lld", need, lim);
    }
  }
  cudaError_t e = cudaMalloc(&s->arena, (size_t)s->arena_bytes);
  if (e != cudaSuccess) {
    delete s;
    return cuda_fail(e, "chunk_stream_create: cudaMalloc(arena)");
  }
  uint8_t* p = static_cast<uint8_t*>(s->arena);
  auto take = [&](int64_t bytes) { auto* r = reinterpret_cast<__nv_bfloat16_raw*>(p); p += bytes; return r; };
  s->ref_k = take(ref_b);
  s->ref_v = take(ref_b);
  for (int i = 0; i < 2; ++i) { s->bnd_k[i] = take(bnd_b); s->bnd_v[i] = take(bnd_b); }
  s->q_rot = take(tok_b);
  s->k_rot = take(tok_b);
  s->o = take(tok_b);
  for (int i = 0; i < 2; ++i) {
    s->anc_k[i] = anc_b ? take(anc_b) : nullptr;
    s->anc_v[i] = anc_b ? take(anc_b) : nullptr;
  }
  s->v_buf = vbuf_b ? take(vbuf_b) : nullptr;
  s->qrope_tab = tab_b ? static_cast<void*>(take(tab_b)) : nullptr;
  for (int i = 0; i < s->n_slots; ++i)
    for (int t = 0; t < 3; ++t) s->in_slot[i][t] = take(tok_b);
  for (int i = 0; i < 2; ++i) s->x_stage[i] = stage_b ? reinterpret_cast<float*>(take(stage_b)) : nullptr;
  if (s->qrope &&
      (rc = rope_q_table_build(s->qrope_tab, c.D, 0, c.F, c.grid_h, c.grid_w, c.rope_base, s->stream))) {
    cudaFree(s->arena);
    delete s;
    return rc;
  }
  if (c.host_io && (rc = host_io_init(s))) {
    host_io_release(s);
    cudaFree(s->arena);
    delete s;
    return rc;
  }
  s->ichunk_index = 0;
  s->cur = 0;
  s->bnd_in_use = 0;
  s->captured = false;
  s->ref_set = false;
  s->chunk_index = 0;
  *out = s;
  return SAVGB_OK;
}

int chunk_stream_set_reference(chunk_stream_t* s, const void* k_ref, const void* v_ref) {
  savgb::ApiRange api_range_("savgb:chunk_stream_set_reference");
  clear_error();
  if (!s || !k_ref || !v_ref) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_set_reference: null argument");
  if (!aligned16(k_ref) || !aligned16(v_ref)) return fail(SAVGB_ERR_ALIGNMENT, "chunk_stream_set_reference: pointers must be 16-byte aligned");
  const chunk_stream_config& c = s->cfg;
  const int64_t per_b = s->n_ref * s->hid;
  RopeArgs a = rope_args(s, k_ref, s->ref_k, per_b, per_b, c.ref_frames, c.ref_t - c.ref_frames + 1);
  int rc = launch_rope(a, s->stream);
  if (rc) return rc;
  SAVGB_CUDA(cudaMemcpyAsync(s->ref_v, v_ref, (size_t)(per_b * c.B * 2), cudaMemcpyDeviceToDevice, s->stream));
  s->ref_set = true;
  s->cur = 0;
  s->bnd_in_use = 0;
  s->captured = false;
  s->chunk_index = 0;
  s->ichunk_index = 0;
  return SAVGB_OK;
}

// The step; with stage >= 0 the W_o update also writes x into that staging copy.
static int step_impl(chunk_stream_t* s, const void* q, const void* k, const void* v, const void* w_o,
                     const float* bias, float* x, float dt, int is_last_step, int stage) {
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step: null handle");
  if (!s->ref_set) return fail(SAVGB_ERR_STATE, "chunk_stream_step: set_reference has not been called");
  if (!q || !k || !v || !w_o || !x) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step: null argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w_o) || !aligned16(x) ||
      (bias && !aligned16(bias)))
    return fail(SAVGB_ERR_ALIGNMENT, "chunk_stream_step: pointers must be 16-byte aligned");
  if (!std::isfinite(dt)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step: dt must be finite");
  const chunk_stream_config& c = s->cfg;
  const int64_t per_b = s->n_tok * s->hid;
  const bool ev = s->have_events;
  s->have_events = false;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[0], s->stream));
  // k is rotated by its own pass; q inside the attention kernel (saving its
  // HBM pass) when the stream's RoPE table fits, else in the same pass as k
  RopeArgs aq = rope_args(s, q, s->q_rot, per_b, per_b, c.F, 0);
  RopeArgs ak = rope_args(s, k, s->k_rot, per_b, per_b, c.F, 0);
  int rc = s->qrope ? launch_rope(ak, s->stream) : launch_rope_pair(aq, ak, s->stream);
  if (rc) return rc;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[1], s->stream));
  AttnSeg segs[3] = {
      {s->ref_k, s->ref_v, s->n_ref},
      {s->bnd_k[s->cur], s->bnd_v[s->cur], s->bnd_in_use},
      {s->k_rot, v, s->n_tok},
  };
  if (s->qrope) {
    QRope r{c.F, c.grid_h, c.grid_w, 0, c.rope_base};
    r.tab = s->qrope_tab;
    r.tab_t_lo = 0;
    r.tab_t_n = c.F;
    rc = launch_attention_qrope(q, c.B, s->n_tok, c.H, c.D, segs, 3, c.softmax_scale, r, s->o, nullptr,
                                s->stream, c.exact_softmax != 0);
  } else {
    rc = launch_attention(s->q_rot, c.B, s->n_tok, c.H, c.D, segs, 3, c.softmax_scale, s->o, nullptr,
                          s->stream, c.exact_softmax != 0);
  }
  if (rc) return rc;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[2], s->stream));
  float* x_copy = nullptr;
  if ((rc = take_stage(s, stage, &x_copy))) return rc;
  rc = launch_out_proj_euler(s->o, w_o, bias, x, c.B * s->n_tok, (int)s->hid, (int)s->hid, dt,
                             nullptr, s->stream, x_copy);
  if (rc) return rc;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[3], s->stream));
  if (is_last_step && s->n_bnd > 0) {
    const int nxt = s->cur ^ 1;
    const int64_t tail = (s->n_tok - s->n_bnd) * s->hid;
    const int64_t bnd_per_b = s->n_bnd * s->hid;
    RopeArgs ab = rope_args(s, static_cast<const __nv_bfloat16_raw*>(k) + tail, s->bnd_k[nxt],
                            per_b, bnd_per_b, c.boundary_frames, -c.boundary_frames);
    if ((rc = launch_rope(ab, s->stream))) return rc;
    SAVGB_CUDA(cudaMemcpy2DAsync(s->bnd_v[nxt], (size_t)bnd_per_b * 2,
                                 static_cast<const __nv_bfloat16_raw*>(v) + tail, (size_t)per_b * 2,
                                 (size_t)bnd_per_b * 2, (size_t)c.B, cudaMemcpyDeviceToDevice,
                                 s->stream));
    s->captured = true;
  } else if (is_last_step) {
    s->captured = true;
  }
  if (is_last_step && c.interp_chunks) {
    // anchors of the interpolation chunks on either side of this N chunk
    const int64_t fr_el = (int64_t)c.grid_h * c.grid_w * s->hid;  // one frame, one session
    const int64_t anc_per_b = 2 * fr_el;
    const int64_t idx = s->chunk_index;
    const int sl_prev = (int)(idx & 1);        // I_idx: this chunk's last frame at t = 0
    const int64_t last = s->n_tok * s->hid - fr_el;
    RopeArgs al = rope_args(s, static_cast<const __nv_bfloat16_raw*>(k) + last, s->anc_k[sl_prev], per_b,
                            anc_per_b, 1, 0);
    if ((rc = launch_rope(al, s->stream))) return rc;
    SAVGB_CUDA(cudaMemcpy2DAsync(s->anc_v[sl_prev], (size_t)anc_per_b * 2,
                                 static_cast<const __nv_bfloat16_raw*>(v) + last, (size_t)per_b * 2,
                                 (size_t)fr_el * 2, (size_t)c.B, cudaMemcpyDeviceToDevice, s->stream));
    if (idx >= 1) {
      const int sl_next = (int)((idx - 1) & 1);  // I_{idx-1}: this chunk's first frame at t = F-1
      RopeArgs af = rope_args(s, k, s->anc_k[sl_next] + fr_el, per_b, anc_per_b, 1, c.F - 1);
      if ((rc = launch_rope(af, s->stream))) return rc;
      SAVGB_CUDA(cudaMemcpy2DAsync(s->anc_v[sl_next] + fr_el, (size_t)anc_per_b * 2, v, (size_t)per_b * 2,
                                   (size_t)fr_el * 2, (size_t)c.B, cudaMemcpyDeviceToDevice, s->stream));
    }
  }
  return SAVGB_OK;
}

int chunk_stream_step(chunk_stream_t* s, const void* q, const void* k, const void* v,
                      const void* w_o, const float* bias, float* x, float dt, int is_last_step) {
  savgb::ApiRange api_range_("savgb:chunk_stream_step");
  clear_error();
  return step_impl(s, q, k, v, w_o, bias, x, dt, is_last_step, -1);
}

int chunk_stream_step_host(chunk_stream_t* s, const void* q_host, const void* k_host, const void* v_host,
                           const void* w_o, const float* bias, float* x, float dt, int is_last_step,
                           float* x_host) {
  savgb::ApiRange api_range_("savgb:chunk_stream_step_host");
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step_host: null handle");
  if (!s->cfg.host_io) return fail(SAVGB_ERR_STATE, "chunk_stream_step_host: the stream was created without host_io");
  if (!s->ref_set) return fail(SAVGB_ERR_STATE, "chunk_stream_step_host: set_reference has not been called");
  if (!q_host || !k_host || !v_host || !w_o || !x)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step_host: null argument");
  if (!std::isfinite(dt)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_step_host: dt must be finite");
  const int slot = s->next_slot;
  const size_t bytes = (size_t)(s->cfg.B * s->n_tok * s->hid * 2);
  // upload into the slot once the step that last read it has finished
  if (s->slot_used[slot]) SAVGB_CUDA(cudaStreamWaitEvent(s->copy_in, s->ev_freed[slot], 0));
  const void* src[3] = {q_host, k_host, v_host};
  for (int t = 0; t < 3; ++t)
    SAVGB_CUDA(cudaMemcpyAsync(s->in_slot[slot][t], src[t], bytes, cudaMemcpyHostToDevice, s->copy_in));
  SAVGB_CUDA(cudaEventRecord(s->ev_loaded[slot], s->copy_in));
  SAVGB_CUDA(cudaStreamWaitEvent(s->stream, s->ev_loaded[slot], 0));
  s->host_used = true;
  const int stage = x_host ? s->next_stage : -1;
  int rc = step_impl(s, s->in_slot[slot][0], s->in_slot[slot][1], s->in_slot[slot][2], w_o, bias, x, dt,
                     is_last_step, stage);
  if (rc) return rc;
  SAVGB_CUDA(cudaEventRecord(s->ev_freed[slot], s->stream));
  s->slot_used[slot] = true;
  s->next_slot = (slot + 1) % s->n_slots;
  if (x_host) {
    // read back the staging copy of x that this step's W_o update wrote; the
    // W_o update that next writes this copy, two host steps later, waits for
    // it, and nothing else does (x itself is not read)
    SAVGB_CUDA(cudaEventRecord(s->ev_step_done, s->stream));
    SAVGB_CUDA(cudaStreamWaitEvent(s->copy_out, s->ev_step_done, 0));
    SAVGB_CUDA(cudaMemcpyAsync(x_host, s->x_stage[stage], (size_t)(s->cfg.B * s->n_tok * s->hid * 4),
                               cudaMemcpyDeviceToHost, s->copy_out));
    SAVGB_CUDA(cudaEventRecord(s->ev_stage_read[stage], s->copy_out));
    SAVGB_CUDA(cudaEventRecord(s->ev_out_done, s->copy_out));
    s->stage_pending[stage] = true;
    s->next_stage = stage ^ 1;
    s->out_pending = true;
  }
  return SAVGB_OK;
}

int chunk_stream_join_copies(chunk_stream_t* s) {
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_join_copies: null handle");
  if (!s->cfg.host_io || !s->host_used) return SAVGB_OK;
  // every upload is already ordered before its step on the stream; the last
  // read-back (ev_out_done follows every earlier one on copy_out) is not
  if (s->out_pending) SAVGB_CUDA(cudaStreamWaitEvent(s->stream, s->ev_out_done, 0));
  s->out_pending = false;
  s->stage_pending[0] = s->stage_pending[1] = false;
  return SAVGB_OK;
}

int chunk_stream_istep(chunk_stream_t* s, const void* q, const void* k, const void* v,
                       const void* w_o, const float* bias, float* x, float dt) {
  savgb::ApiRange api_range_("savgb:chunk_stream_istep");
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_istep: null handle");
  const chunk_stream_config& c = s->cfg;
  if (!c.interp_chunks) return fail(SAVGB_ERR_STATE, "chunk_stream_istep: the stream was created without interp_chunks");
  if (!s->ref_set) return fail(SAVGB_ERR_STATE, "chunk_stream_istep: set_reference has not been called");
  if (!q || !k || !v || !w_o || !x) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_istep: null argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(w_o) || !aligned16(x) ||
      (bias && !aligned16(bias)))
    return fail(SAVGB_ERR_ALIGNMENT, "chunk_stream_istep: pointers must be 16-byte aligned");
  if (!std::isfinite(dt)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_istep: dt must be finite");
  if (s->chunk_index > s->ichunk_index + 2) s->ichunk_index = s->chunk_index - 2;  // anchors of older ones are gone
  if (s->captured && s->chunk_index == s->ichunk_index + 2)
    return fail(SAVGB_ERR_STATE, "chunk_stream_istep: I chunk %lld must run before the last step of N chunk %lld",
                (long long)s->ichunk_index, (long long)s->chunk_index);
  if (s->chunk_index < s->ichunk_index + 2)
    return fail(SAVGB_ERR_STATE, "chunk_stream_istep: I chunk %lld needs N chunks %lld and %lld finished (%lld are)",
                (long long)s->ichunk_index, (long long)s->ichunk_index, (long long)s->ichunk_index + 1,
                (long long)s->chunk_index);
  const int64_t fr = (int64_t)c.grid_h * c.grid_w;
  const int64_t n_int = (c.F - 2) * fr;
  const int64_t per_b = n_int * s->hid;
  RopeArgs aq = rope_args(s, q, s->q_rot, per_b, per_b, c.F - 2, 1);
  RopeArgs ak = rope_args(s, k, s->k_rot, per_b, per_b, c.F - 2, 1);
  int rc = s->qrope ? launch_rope(ak, s->stream) : launch_rope_pair(aq, ak, s->stream);
  if (rc) return rc;
  const int sl = (int)(s->ichunk_index & 1);
  AttnSeg segs[3] = {
      {s->ref_k, s->ref_v, s->n_ref},
      {s->anc_k[sl], s->anc_v[sl], 2 * fr},
      {s->k_rot, v, n_int},
  };
  if (s->qrope) {
    // the interior frames sit at t = 1 .. F-2 of the stream's table
    QRope r{c.F - 2, c.grid_h, c.grid_w, 1, c.rope_base};
    r.tab = s->qrope_tab;
    r.tab_t_lo = 0;
    r.tab_t_n = c.F;
    rc = launch_attention_qrope(q, c.B, n_int, c.H, c.D, segs, 3, c.softmax_scale, r, s->o, nullptr, s->stream,
                                c.exact_softmax != 0);
  } else {
    rc = launch_attention(s->q_rot, c.B, n_int, c.H, c.D, segs, 3, c.softmax_scale, s->o, nullptr, s->stream,
                          c.exact_softmax != 0);
  }
  if (rc) return rc;
  return launch_out_proj_euler(s->o, w_o, bias, x, c.B * n_int, (int)s->hid, (int)s->hid, dt, nullptr,
                               s->stream);
}

int chunk_stream_end_ichunk(chunk_stream_t* s) {
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_end_ichunk: null handle");
  if (!s->cfg.interp_chunks) return fail(SAVGB_ERR_STATE, "chunk_stream_end_ichunk: no interpolation chunks");
  if (s->chunk_index < s->ichunk_index + 2)
    return fail(SAVGB_ERR_STATE, "chunk_stream_end_ichunk: I chunk %lld has not started", (long long)s->ichunk_index);
  s->ichunk_index += 1;
  return SAVGB_OK;
}

int chunk_stream_ichunk_index(const chunk_stream_t* s, int64_t* index) {
  clear_error();
  if (!s || !index) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_ichunk_index: null argument");
  *index = s->ichunk_index;
  return SAVGB_OK;
}

int chunk_stream_block_step(chunk_stream_t* s, const void* w_qkv, const void* w_o, const float* bias,
                            float* x, float dt, int is_last_step) {
  savgb::ApiRange api_range_("savgb:chunk_stream_block_step");
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_block_step: null handle");
  const chunk_stream_config& c = s->cfg;
  if (!c.qkv_block) return fail(SAVGB_ERR_STATE, "chunk_stream_block_step: the stream was created without qkv_block");
  if (!s->ref_set) return fail(SAVGB_ERR_STATE, "chunk_stream_block_step: set_reference has not been called");
  if (!w_qkv || !w_o || !x) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_block_step: null argument");
  if (!aligned16(w_qkv) || !aligned16(w_o) || !aligned16(x) || (bias && !aligned16(bias)))
    return fail(SAVGB_ERR_ALIGNMENT, "chunk_stream_block_step: pointers must be 16-byte aligned");
  if (!std::isfinite(dt)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_block_step: dt must be finite");
  const bool ev = s->have_events;
  s->have_events = false;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[0], s->stream));
  const int64_t M = (int64_t)c.B * s->n_tok;
  void* xb = s->o;  // the bf16 copy of x is consumed by the projection before attention writes o
  int rc = launch_to_bf16(x, xb, M * s->hid, s->stream);
  if (rc) return rc;
  const int nxt = s->cur ^ 1;
  const bool capture = is_last_step && s->n_bnd > 0;
  QkvArgs qa{xb, w_qkv, s->q_rot, s->k_rot, s->v_buf, capture ? s->bnd_k[nxt] : nullptr, s->n_bnd, c.B,
             s->n_tok, c.H, c.D, c.F, c.grid_h, c.grid_w, 0, c.rope_base};
  if ((rc = validate_qkv(qa))) return rc;
  if ((rc = launch_qkv_rope(qa, s->stream))) return rc;
  if (capture) {
    // the boundary: the projected k (stored unrotated by the projection) and v
    // of the last frames, k rotated in place to t = -T_b .. -1
    const int64_t bnd_per_b = s->n_bnd * s->hid;
    RopeArgs ab = rope_args(s, s->bnd_k[nxt], s->bnd_k[nxt], bnd_per_b, bnd_per_b, c.boundary_frames,
                            -c.boundary_frames);
    if ((rc = launch_rope(ab, s->stream))) return rc;
    const int64_t per_b = s->n_tok * s->hid;
    SAVGB_CUDA(cudaMemcpy2DAsync(s->bnd_v[nxt], (size_t)bnd_per_b * 2, s->v_buf + (per_b - bnd_per_b),
                                 (size_t)per_b * 2, (size_t)bnd_per_b * 2, (size_t)c.B, cudaMemcpyDeviceToDevice,
                                 s->stream));
  }
  if (is_last_step) s->captured = true;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[1], s->stream));
  AttnSeg segs[3] = {
      {s->ref_k, s->ref_v, s->n_ref},
      {s->bnd_k[s->cur], s->bnd_v[s->cur], s->bnd_in_use},
      {s->k_rot, s->v_buf, s->n_tok},
  };
  if ((rc = launch_attention(s->q_rot, c.B, s->n_tok, c.H, c.D, segs, 3, c.softmax_scale, s->o, nullptr,
                             s->stream, c.exact_softmax != 0)))
    return rc;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[2], s->stream));
  if ((rc = launch_out_proj_euler(s->o, w_o, bias, x, M, (int)s->hid, (int)s->hid, dt, nullptr, s->stream)))
    return rc;
  if (ev) SAVGB_CUDA(cudaEventRecord(s->step_events[3], s->stream));
  return SAVGB_OK;
}

int chunk_stream_end_chunk(chunk_stream_t* s) {
  savgb::ApiRange api_range_("savgb:chunk_stream_end_chunk");
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_end_chunk: null handle");
  if (!s->captured)
    return fail(SAVGB_ERR_STATE, "chunk_stream_end_chunk: no step of this chunk had is_last_step set");
  if (s->n_bnd > 0) {
    s->cur ^= 1;
    s->bnd_in_use = s->n_bnd;
  }
  s->captured = false;
  s->chunk_index += 1;
  return SAVGB_OK;
}

int chunk_stream_set_step_events(chunk_stream_t* s, void* const* events) {
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_set_step_events: null handle");
  if (!events) {
    s->have_events = false;
    return SAVGB_OK;
  }
  for (int i = 0; i < 4; ++i) {
    if (!events[i]) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_set_step_events: null event %d", i);
    s->step_events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  s->have_events = true;
  return SAVGB_OK;
}

int chunk_stream_sync(chunk_stream_t* s) {
  savgb::ApiRange api_range_("savgb:chunk_stream_sync");
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_sync: null handle");
  if (s->cfg.host_io) {
    SAVGB_CUDA(cudaStreamSynchronize(s->copy_in));
    SAVGB_CUDA(cudaStreamSynchronize(s->copy_out));
    s->out_pending = false;
    s->stage_pending[0] = s->stage_pending[1] = false;
    s->host_used = false;
  }
  return savgb_device_check(s->stream);
}

int chunk_stream_info(const chunk_stream_t* s, int64_t* chunk_index, int64_t* boundary_tokens,
                      int64_t* arena_bytes, const void** boundary_k, const void** boundary_v) {
  clear_error();
  if (!s) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_info: null handle");
  if (chunk_index) *chunk_index = s->chunk_index;
  if (boundary_tokens) *boundary_tokens = s->bnd_in_use;
  if (arena_bytes) *arena_bytes = s->arena_bytes;
  if (boundary_k) *boundary_k = s->bnd_in_use ? s->bnd_k[s->cur] : nullptr;
  if (boundary_v) *boundary_v = s->bnd_in_use ? s->bnd_v[s->cur] : nullptr;
  return SAVGB_OK;
}

int chunk_stream_fused_q_rope(const chunk_stream_t* s, int* fused) {
  clear_error();
  if (!s || !fused) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_fused_q_rope: null argument");
  *fused = s->qrope ? 1 : 0;
  return SAVGB_OK;
}

int chunk_stream_export_state(chunk_stream_t* s, void* buf, size_t cap, size_t* size_out) {
  savgb::ApiRange api_range_("savgb:chunk_stream_export_state");
  clear_error();
  if (!s || !size_out) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_export_state: null argument");
  const int64_t fr = (int64_t)s->cfg.grid_h * s->cfg.grid_w;
  const int64_t anc_bytes = s->cfg.interp_chunks ? 2 * fr * s->hid * 2 * s->cfg.B : 0;  // one slot, K or V
  const int64_t payload = 2 * s->bnd_in_use * s->hid * 2 * s->cfg.B + 4 * anc_bytes;
  const size_t total = sizeof(StateHeader) + (size_t)payload;
  *size_out = total;
  if (!buf) return SAVGB_OK;
  if (cap < total) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_export_state: buffer of %zu bytes < %zu", cap, total);
  StateHeader h{};
  h.magic = kStateMagic;
  const chunk_stream_config& c = s->cfg;
  h.B = c.B; h.H = c.H; h.D = c.D; h.F = c.F; h.grid_h = c.grid_h; h.grid_w = c.grid_w;
  h.boundary_frames = c.boundary_frames;
  h.interp = c.interp_chunks ? 1 : 0;
  h.chunk_index = s->chunk_index;
  h.bnd_in_use = s->bnd_in_use;
  h.payload_bytes = payload;
  h.ichunk_index = s->ichunk_index;
  memcpy(buf, &h, sizeof(h));
  uint8_t* dst = static_cast<uint8_t*>(buf) + sizeof(h);
  const size_t half = (size_t)(s->bnd_in_use * s->hid * 2 * c.B);
  if (half > 0) {
    SAVGB_CUDA(cudaMemcpyAsync(dst, s->bnd_k[s->cur], half, cudaMemcpyDeviceToHost, s->stream));
    SAVGB_CUDA(cudaMemcpyAsync(dst + half, s->bnd_v[s->cur], half, cudaMemcpyDeviceToHost, s->stream));
  }
  dst += 2 * half;
  for (int i = 0; i < 2 && anc_bytes > 0; ++i) {
    SAVGB_CUDA(cudaMemcpyAsync(dst, s->anc_k[i], (size_t)anc_bytes, cudaMemcpyDeviceToHost, s->stream));
    SAVGB_CUDA(cudaMemcpyAsync(dst + anc_bytes, s->anc_v[i], (size_t)anc_bytes, cudaMemcpyDeviceToHost, s->stream));
    dst += 2 * anc_bytes;
  }
  SAVGB_CUDA(cudaStreamSynchronize(s->stream));
  return SAVGB_OK;
}

int chunk_stream_import_state(chunk_stream_t* s, const void* buf, size_t size) {
  savgb::ApiRange api_range_("savgb:chunk_stream_import_state");
  clear_error();
  if (!s || !buf) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_import_state: null argument");
  if (size < sizeof(StateHeader)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_import_state: truncated state");
  StateHeader h;
  memcpy(&h, buf, sizeof(h));
  const chunk_stream_config& c = s->cfg;
  if (h.magic != kStateMagic || h.B != c.B || h.H != c.H || h.D != c.D || h.F != c.F ||
      h.grid_h != c.grid_h || h.grid_w != c.grid_w || h.boundary_frames != c.boundary_frames ||
      h.interp != (c.interp_chunks ? 1 : 0))
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_import_state: state of another configuration");
  const int64_t fr = (int64_t)c.grid_h * c.grid_w;
  const int64_t anc_bytes = c.interp_chunks ? 2 * fr * s->hid * 2 * c.B : 0;
  if ((h.bnd_in_use != 0 && h.bnd_in_use != s->n_bnd) ||
      h.payload_bytes != 2 * h.bnd_in_use * s->hid * 2 * c.B + 4 * anc_bytes ||
      size != sizeof(StateHeader) + (size_t)h.payload_bytes || h.chunk_index < 0 || h.ichunk_index < 0)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_stream_import_state: inconsistent sizes");
  if (!s->ref_set) return fail(SAVGB_ERR_STATE, "chunk_stream_import_state: set_reference first");
  const uint8_t* src = static_cast<const uint8_t*>(buf) + sizeof(h);
  const size_t half = (size_t)(h.bnd_in_use * s->hid * 2 * c.B);
  if (half > 0) {
    SAVGB_CUDA(cudaMemcpyAsync(s->bnd_k[s->cur], src, half, cudaMemcpyHostToDevice, s->stream));
    SAVGB_CUDA(cudaMemcpyAsync(s->bnd_v[s->cur], src + half, half, cudaMemcpyHostToDevice, s->stream));
  }
  src += 2 * half;
  for (int i = 0; i < 2 && anc_bytes > 0; ++i) {
    SAVGB_CUDA(cudaMemcpyAsync(s->anc_k[i], src, (size_t)anc_bytes, cudaMemcpyHostToDevice, s->stream));
    SAVGB_CUDA(cudaMemcpyAsync(s->anc_v[i], src + anc_bytes, (size_t)anc_bytes, cudaMemcpyHostToDevice, s->stream));
    src += 2 * anc_bytes;
  }
  SAVGB_CUDA(cudaStreamSynchronize(s->stream));
  s->bnd_in_use = h.bnd_in_use;
  s->chunk_index = h.chunk_index;
  s->ichunk_index = h.ichunk_index;
  s->captured = false;
  return SAVGB_OK;
}

int chunk_stream_destroy(chunk_stream_t* s) {
  savgb::ApiRange api_range_("savgb:chunk_stream_destroy");
  clear_error();
  if (!s) return SAVGB_OK;
  cudaError_t e1 = cudaStreamSynchronize(s->stream);
  if (s->cfg.host_io) host_io_release(s);
  cudaError_t e2 = cudaFree(s->arena);
  delete s;
  if (e1 != cudaSuccess) return cuda_fail(e1, "chunk_stream_destroy: cudaStreamSynchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "chunk_stream_destroy: cudaFree");
  return SAVGB_OK;
}

}  // extern "C"
