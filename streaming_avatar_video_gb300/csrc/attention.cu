// Chunk attention on the sm_103a tensor cores (tcgen05 + tensor memory + TMA).
//
// Queries of the current chunk attend over up to three key/value segments,
// [static reference | previous chunk's boundary | current chunk] (HeyGen,
// "Avatar inference at scale", sections "The underlying model architecture"
// and "The streaming framework and pipeline loop").  O = softmax(s Q K^T) V
// per (batch, head), no mask.
//
// Design (one CTA = two 128-row query tiles of one (batch, head)):
//   warp 0      TMA producer of Q (once) and of the K tiles of the
//               concatenated segments (3-stage ring); warp 2 that of the V
//               tiles (2-stage ring).  Both run their loop warp-wide and one
//               elected lane issues the copies.
//   warp 1      allocates 512 TMEM columns and runs the MMA issue loop; one
//               elected lane issues every tcgen05.mma.
//   warp 3      checks that each key tile's V and the next K have landed and
//               adds one arrival to the P barrier of tile 0.
//   warps 4-7   softmax of query tile 0, warps 8-11 of query tile 1; thread =
//               one query row (TMEM lane), so row max and sum need no shuffle.
// Registers: the block launches with 168 per thread; the first warpgroup
// gives back down to 88 and the two softmax warpgroups take 208 each
// (setmaxnreg), so a thread holds a whole 128-column score row without spills.
// TMEM columns: S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [256+D,256+2D).
// P (bf16) overwrites the first 64 columns of its S and feeds the PV product
// straight from TMEM.  The two query tiles alternate so that the tensor core
// works on one tile's QK^T / PV while the other tile's softmax runs.
// tcgen05.mma issue is nearly synchronous with execution (the unit holds
// about one instruction ahead), so every clock the issuing thread spends
// between MMAs idles the tensor core: the issue loop has two wait points per
// key tile (P of tile 0, P of tile 1) and no other work.  A satisfied
// mbarrier try_wait still costs it ~60 clocks, so the check that V(j) and
// K(j+1) have landed is made by warp 3, which arrives on P of tile 0 too.
// The running max is updated lazily (only when it grows by more than 2^8 in
// probability), and O is rescaled in TMEM by the softmax warps when it is.
// The probabilities come from one packed bf16x2 exp2 per two scores (their
// exponents rounded to bf16), which yields the bf16 P operand directly; the
// row sums add those same bf16 values in fp32.  When the log-sum-exp output is
// asked for, an instantiation with fp32 exponentials and exact sums runs.
// At the end each softmax warp normalises its 32 rows of O into the Q tile's
// shared memory (free by then) and writes them with tensor-map stores.
// Built with ROPE_Q (chunk_attention_qrope) the kernel takes unrotated
// queries: the block's part of a cos/sin table arrives from global memory with
// Q, and the softmax threads rotate one query row each in shared memory before
// the first MMA.
// Every wait is bounded; on a timeout the block records it in the device
// error word and every role leaves its loop.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "common.h"
#include "ptx.cuh"

namespace savgb {
namespace {

constexpr int kThreads = 384;
constexpr int kRegsLow = 88;     // producer / MMA warpgroup after setmaxnreg.dec
constexpr int kRegsHigh = 208;  // softmax warpgroups after setmaxnreg.inc
// the split must fit the block's launch pool: kThreads * launch registers
constexpr int kRegPoolNeeded = 128 * kRegsLow + 256 * kRegsHigh;
constexpr int kBlockQ = 256;  // two 128-row tiles
constexpr int kTileKV = 128;
// a tile whose probabilities against the running max sum to more than this
// (2^8) moves the max; below it no probability exceeds 2^8
constexpr float kTileSumLimit = 256.0f;
// softmax scales above this multiple of 1/sqrt(D) take fp32 exponentials
constexpr float kExactScaleRatio = 1.25f;
// K / V ring depths: 128-row tiles of 32 KiB (D=128) or 16 KiB (D=64)
#ifndef SAVGB_ATTN_KS128
#define SAVGB_ATTN_KS128 3
#endif
#ifndef SAVGB_ATTN_VS128
#define SAVGB_ATTN_VS128 2
#endif
constexpr int kStagesK128 = SAVGB_ATTN_KS128, kStagesV128 = SAVGB_ATTN_VS128;
constexpr int kStagesK64 = 4, kStagesV64 = 4;

struct AttnMaps {
  CUtensorMap q;
  CUtensorMap k[3];
  CUtensorMap v[3];
  CUtensorMap o;  // 32-row boxes: one softmax warp's rows
};

struct AttnParams {
  int n_q, H, n_tiles;
  int seg_tiles[3];
  int seg_len[3];
  float scale_log2;
  float* lse;
  DeviceErrorWord* err;
  // 3D RoPE of the queries, applied in shared memory when the kernel is built
  // with ROPE_Q: query token n sits at (t0 + n/(gh*gw), (n/gw)%gh, n%gw).
  // The cos/sin table in global memory is [t rows (tab_t_n from tab_t_lo) |
  // h section (tab_h_sec entries) | w section]; a block copies its own t rows
  // (at most tab_t_rows) and the h and w sections into shared memory.
  int gh, gw, t0;
  const float2* rope_tab;
  int tab_t_lo, tab_t_n;
  int tab_t_rows;      // time rows one block's 256 queries can span
  int tab_h_sec;       // entries of the h section (padded to 16 bytes)
  int tab_hw_entries;  // entries of the h and w sections
  // failure-path test hook (savgb_arm_wait_fault): key tile whose copy the K
  // producer of block (0, 0, 0) skips (-1: none), and the limit of every wait
  int fault_tile;
  uint64_t wait_limit_ns;
};

template <int D, int KS, int VS>
struct Layout {
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row tile, D/64 swizzled column blocks
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + KS * kTileBytes;
  static constexpr int kBar = kV + VS * kTileBytes;
  // barriers: Q full, K full/empty per stage, V full/empty per stage,
  // S full / P full / O done per query tile, MMA drain
  static constexpr int kQFull = 0;
  static constexpr int kKFull = 1;
  static constexpr int kKEmpty = kKFull + KS;
  static constexpr int kVFull = kKEmpty + KS;
  static constexpr int kVEmpty = kVFull + VS;
  static constexpr int kSFull = kVEmpty + VS;
  static constexpr int kP = kSFull + 2;  // a tile's probabilities written to TMEM
  static constexpr int kODone = kP + 2;
  static constexpr int kDrain = kODone + 2;
  static constexpr int kQReady = kDrain + 1;  // queries rotated in place (ROPE_Q)
  static constexpr int kNumBars = kQReady + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTab = (kMisc + 16 + 127) / 128 * 128;  // cos/sin tables of the query RoPE (ROPE_Q only)
  static constexpr int kBytes = kTab;
  // request at least 120 KiB so two blocks never share an SM (each holds all 512 TMEM columns)
  static constexpr int kDynSmem = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
  static_assert(kBytes + 1024 <= 227 * 1024, "shared memory budget");
};

// Key tile j of the concatenated segments: its segment, first row and valid
// rows.  Only constant indices into the parameters, so nothing is copied to
// local memory.
__device__ __forceinline__ void tile_of(const AttnParams& p, int j, int& seg, int& row0, int& valid) {
  const int e0 = p.seg_tiles[0], e1 = e0 + p.seg_tiles[1];
  seg = j < e0 ? 0 : (j < e1 ? 1 : 2);
  row0 = (j - (seg == 0 ? 0 : (seg == 1 ? e0 : e1))) * kTileKV;
  const int len = seg == 0 ? p.seg_len[0] : (seg == 1 ? p.seg_len[1] : p.seg_len[2]);
  const int rest = len - row0;
  valid = rest < kTileKV ? rest : kTileKV;
}

__device__ __forceinline__ void give_up(const AttnParams& p, volatile int* abort, unsigned code) {
  if (atomicExch(const_cast<int*>(abort), 1) == 0) {
    atomicOr(&p.err->flags, kErrAttnWait);
    atomicCAS(&p.err->where, 0u, code);
  }
}

// Channel pairs of each RoPE axis: D/2 pairs, a third each (rounded down)
// for h and w and the rest for t, in the order [t | h | w].
template <int D>
struct RopeSplit {
  static constexpr int kP = D / 2, kH = kP / 3, kW = kP / 3, kT = kP - 2 * (kP / 3);
};

__host__ __device__ constexpr int64_t even_up(int64_t n) { return (n + 1) & ~static_cast<int64_t>(1); }

// The cos/sin table of the query RoPE in global memory: float2 (cos, sin)
// for [n_t time rows from t_lo | grid_h rows | grid_w rows] x their axis's
// pairs, each section padded to an even number of entries (16 bytes).
// Pair j of an axis with P pairs turns at base^(-j/P) per unit of position.
template <int D>
__global__ void rope_q_table_kernel(float2* tab, int t_lo, int n_t, int gh, int gw, float log2_base) {
  using R = RopeSplit<D>;
  const int n_tt = n_t * R::kT, n_h = gh * R::kH, n_w = gw * R::kW;
  const int h_off = static_cast<int>(even_up(n_tt));
  const int w_off = h_off + static_cast<int>(even_up(n_h));
  const int total = w_off + static_cast<int>(even_up(n_w));
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int pos, j, P;
    if (i < n_tt) { pos = t_lo + i / R::kT; j = i % R::kT; P = R::kT; }
    else if (i >= h_off && i < h_off + n_h) { const int k = i - h_off; pos = k / R::kH; j = k % R::kH; P = R::kH; }
    else if (i >= w_off && i < w_off + n_w) { const int k = i - w_off; pos = k / R::kW; j = k % R::kW; P = R::kW; }
    else { tab[i] = make_float2(1.f, 0.f); continue; }  // padding, never read
    const float omega = exp2f(-static_cast<float>(j) / static_cast<float>(P) * log2_base);
    float sn, cs;
    sincosf(static_cast<float>(pos) * omega, &sn, &cs);
    tab[i] = make_float2(cs, sn);
  }
}

// Rotates, in place, one query row of the two swizzled Q tiles: row r of the
// block (tile r/128), token q = q0 + r, by table lookup.
template <int D>
__device__ __forceinline__ void rope_q_row(uint8_t* sQ, int tile_bytes, const float2* tab, int r, int q0,
                                           const AttnParams& p) {
  const int x = r >> 7, rr = r & 127;
  const int hw = p.gh * p.gw;
  const int q = q0 + r;
  const int tt = q / hw - q0 / hw;  // time row within the block's table
  const int r2 = q % hw;
  const int hh = r2 / p.gw;
  const int ww = r2 - hh * p.gw;
  using R = RopeSplit<D>;
  const float2* tr = tab + tt * R::kT;
  const float2* hr = tab + p.tab_t_rows * R::kT + hh * R::kH - R::kT;
  const float2* wr = tab + p.tab_t_rows * R::kT + p.tab_h_sec + ww * R::kW - R::kT - R::kH;
  #pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    #pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint4* cell = reinterpret_cast<uint4*>(sQ + x * tile_bytes + c * 16384 + rr * 128 + ((j ^ (rr & 7)) << 4));
      uint4 v = *cell;
      uint32_t w0 = v.x, w1 = v.y, w2 = v.z, w3 = v.w;
      #define SAVGB_QROT(W, U) { const int pr = c * 32 + 4 * j + (U);                                   \
        const float2 cs = pr < R::kT ? tr[pr] : (pr < R::kT + R::kH ? hr[pr] : wr[pr]);              \
        __nv_bfloat162 e = *reinterpret_cast<__nv_bfloat162*>(&W);                                    \
        const float a = __low2float(e), b = __high2float(e);                                          \
        __nv_bfloat162 o2 = __floats2bfloat162_rn(a * cs.x - b * cs.y, a * cs.y + b * cs.x);          \
        W = *reinterpret_cast<uint32_t*>(&o2); }
      SAVGB_QROT(w0, 0) SAVGB_QROT(w1, 1) SAVGB_QROT(w2, 2) SAVGB_QROT(w3, 3)
      #undef SAVGB_QROT
      *cell = make_uint4(w0, w1, w2, w3);
    }
  }
}

// One thread's row of a 128-column score tile from tensor memory; columns
// at or past `valid` (a segment's ragged tail) read as -inf.
__device__ __forceinline__ void load_scores(uint32_t tS, uint32_t (&sr)[128], int valid) {
  uint32_t (&lo)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sr[0]);
  uint32_t (&hi)[64] = *reinterpret_cast<uint32_t(*)[64]>(&sr[64]);
  dev::tmem_ld64(tS, lo);
  dev::tmem_ld64(tS + 64, hi);
  if (valid < kTileKV) {
    #pragma unroll
    for (int c = 0; c < kTileKV; ++c)
      if (c >= valid) sr[c] = __float_as_uint(-INFINITY);
  }
}

// Row max: a shallow tree of 3-input maxes (128 -> 43 -> 15 -> 5 -> 2 -> 1).
__device__ __forceinline__ float row_max(const float* s) {
  float t1[43];
  #pragma unroll
  for (int i = 0; i < 42; ++i) t1[i] = dev::fmax3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
  t1[42] = fmaxf(s[126], s[127]);
  float t2[15];
  #pragma unroll
  for (int i = 0; i < 14; ++i) t2[i] = dev::fmax3(t1[3 * i], t1[3 * i + 1], t1[3 * i + 2]);
  t2[14] = t1[42];
  float t3[5];
  #pragma unroll
  for (int i = 0; i < 5; ++i) t3[i] = dev::fmax3(t2[3 * i], t2[3 * i + 1], t2[3 * i + 2]);
  return fmaxf(dev::fmax3(t3[0], t3[1], t3[2]), fmaxf(t3[3], t3[4]));
}

// The tile's probabilities p = 2^(s * sl2 - m) as 64 bf16x2 words (the PV
// operand), nm = -m, and their sum in (l0, l1).
// EXACT_L: fp32 exponentials (one MUFU operation per score) summed exactly,
// as the log-sum-exp output needs; otherwise one packed bf16x2 exponential
// per two scores on the exponents rounded to bf16, whose result is already
// the operand; the sum adds those bf16 values two words at a time in bf16x2
// and then in fp32 (~0.3 % low on average against fp32 exponentials, which
// cancels in O).
template <bool EXACT_L>
__device__ __forceinline__ void tile_exp(const float* s, float sl2, float nm, uint32_t (&pk)[64], float& l0,
                                         float& l1) {
  if constexpr (EXACT_L) {
    #pragma unroll
    for (int i = 0; i < 64; ++i) {
      float y0, y1;
      dev::ffma2(y0, y1, s[2 * i], s[2 * i + 1], sl2, nm);
      const float p0 = dev::ex2_approx(y0);
      const float p1 = dev::ex2_approx(y1);
      dev::fadd2(l0, l1, p0, p1);
      pk[i] = dev::pack_bf16x2(p0, p1);
    }
  } else {
    #pragma unroll
    for (int i = 0; i < 64; i += 2) {
      float y0, y1, y2, y3;
      dev::ffma2(y0, y1, s[2 * i], s[2 * i + 1], sl2, nm);
      dev::ffma2(y2, y3, s[2 * i + 2], s[2 * i + 3], sl2, nm);
      pk[i] = dev::ex2_bf16x2(dev::pack_bf16x2(y0, y1));
      pk[i + 1] = dev::ex2_bf16x2(dev::pack_bf16x2(y2, y3));
      // two words' probabilities added pairwise in bf16x2, then widened
      // exactly into the fp32 sums: half the fp32 additions, one more bf16
      // rounding per pair of probabilities in the denominator only
      dev::add_bf16x2_to_f32(l0, l1, dev::add_bf16x2(pk[i], pk[i + 1]));
    }
  }
}

// EXACT_L: the row sums come from fp32 probabilities (one MUFU operation per
// score), as the log-sum-exp output needs; otherwise from the bf16 ones of
// the packed exponential (one operation per two scores), whose rounding
// leaves the sum ~0.3 % low on average but matches the P the PV product uses.
template <int D, int KS, int VS, bool ROPE_Q, bool EXACT_L>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ AttnParams p) {
  using L = Layout<D, KS, VS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = dev::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * kBlockQ;

  if (tid == 0) {
    dev::mbar_init(&bars[L::kQFull], 1);
    for (int s = 0; s < KS; ++s) {
      dev::mbar_init(&bars[L::kKFull + s], 1);
      dev::mbar_init(&bars[L::kKEmpty + s], 1);
    }
    for (int s = 0; s < VS; ++s) {
      dev::mbar_init(&bars[L::kVFull + s], 1);
      dev::mbar_init(&bars[L::kVEmpty + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      dev::mbar_init(&bars[L::kSFull + x], 1);
      // one elected lane per softmax warp; for tile 0 also warp 3 (V and K landed)
      dev::mbar_init(&bars[L::kP + x], x == 0 ? 5 : 4);
      dev::mbar_init(&bars[L::kODone + x], 1);
    }
    dev::mbar_init(&bars[L::kDrain], 1);
    dev::mbar_init(&bars[L::kQReady], 8);  // one elected lane per softmax warp
    *abort = 0;
    dev::fence_barrier_init();
  }
  if (warp == 1) {
    dev::tmem_alloc(tmem_slot, 512);
    dev::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    dev::tma_prefetch_desc(&maps.q);
    for (int s = 0; s < 3; ++s) {
      if (p.seg_tiles[s] > 0) {
        dev::tma_prefetch_desc(&maps.k[s]);
        dev::tma_prefetch_desc(&maps.v[s]);
      }
    }
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n = p.n_tiles;
  // the set-up above overlaps the previous kernel of the stream (RoPE of q, k)
  dev::griddep_launch_dependents();
  dev::griddep_wait();

  if (warp < 4) {
    dev::setmaxnreg_dec<kRegsLow>();
    if (warp == 0 || warp == 2) {
      // ------------------------------------------- producers: K (warp 0), V (warp 2)
      // the whole warp runs the loop; one elected lane issues the copies
      const bool elected = dev::elect_one();
      const bool is_k = warp == 0;
      const int stages = is_k ? KS : VS;
      uint8_t* ring = smem + (is_k ? L::kK : L::kV);
      uint64_t* full = &bars[is_k ? L::kKFull : L::kVFull];
      uint64_t* empty = &bars[is_k ? L::kKEmpty : L::kVEmpty];
      // test hook: block (0, 0, 0) leaves one key tile uncopied (fault_tile < 0: never)
      const int skip = (is_k && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) ? p.fault_tile : -1;
      if (is_k && elected) {
        uint8_t* sQ = smem + L::kQ;
        if constexpr (ROPE_Q) {
          // this block's time rows and the h and w sections of the RoPE table,
          // on the Q barrier
          using R = RopeSplit<D>;
          const int r0 = p.t0 + q0 / (p.gh * p.gw) - p.tab_t_lo;
          const int rows = min(p.tab_t_rows, p.tab_t_n - r0);
          const uint32_t tb = static_cast<uint32_t>(rows * R::kT * 8);
          const uint32_t hb = static_cast<uint32_t>(p.tab_hw_entries * 8);
          float2* st = reinterpret_cast<float2*>(smem + L::kTab);
          dev::mbar_arrive_expect_tx(&bars[L::kQFull], 2 * L::kTileBytes + tb + hb);
          dev::bulk_load(st, p.rope_tab + r0 * R::kT, tb, &bars[L::kQFull]);
          dev::bulk_load(st + p.tab_t_rows * R::kT, p.rope_tab + p.tab_t_n * R::kT, hb, &bars[L::kQFull]);
        } else {
          dev::mbar_arrive_expect_tx(&bars[L::kQFull], 2 * L::kTileBytes);
        }
        #pragma unroll
        for (int x = 0; x < 2; ++x)
          #pragma unroll
          for (int c = 0; c < D / 64; ++c)
            dev::tma_load_4d(sQ + x * L::kTileBytes + c * 16384, &maps.q, &bars[L::kQFull], c * 64, h,
                             q0 + x * 128, b);
      }
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        int seg, row0, valid;
        tile_of(p, j, seg, row0, valid);
        const int st = j % stages;
        const uint32_t use = j / stages;
        if (j >= stages && !__all_sync(0xffffffffu, dev::mbar_wait(&empty[st], (use - 1) & 1, abort, p.wait_limit_ns))) {
          if (elected) give_up(p, abort, is_k ? 1 : 2);
          break;
        }
        if (elected && j != skip) {
          dev::mbar_arrive_expect_tx(&full[st], L::kTileBytes);
          #pragma unroll
          for (int c = 0; c < D / 64; ++c)
            dev::tma_load_4d(ring + st * L::kTileBytes + c * 16384,
                             is_k ? (seg == 0 ? &maps.k[0] : (seg == 1 ? &maps.k[1] : &maps.k[2]))
                                  : (seg == 0 ? &maps.v[0] : (seg == 1 ? &maps.v[1] : &maps.v[2])),
                             &full[st], c * 64, h, row0, b);
        }
        issued = j + 1;
      }
      // drain: every issued copy has landed before the block may exit
      volatile int never = 0;
      if (is_k) dev::mbar_wait(&bars[L::kQFull], 0, &never, p.wait_limit_ns);
      for (int t = (issued > stages ? issued - stages : 0); t < issued; ++t)
        dev::mbar_wait(&full[t % stages], (t / stages) & 1, &never, p.wait_limit_ns);
    } else if (warp == 3) {
      // ------------------------------------------------ V/K landing checks
      // For every key tile j: V(j) and K(j+1) have landed, then one arrival
      // on P of tile 0, so the MMA issuer's wait on that P covers them (a
      // satisfied try_wait costs the issuer ~60 clocks).  The next arrival
      // waits until this phase has completed, so it never counts towards it.
      const bool elected = dev::elect_one();
      for (int j = 0; j < n; ++j) {
        const bool kv = j + 1 < n ? dev::mbar_wait2(&bars[L::kVFull + j % VS], (j / VS) & 1,
                                                    &bars[L::kKFull + (j + 1) % KS], ((j + 1) / KS) & 1, abort, p.wait_limit_ns)
                                  : dev::mbar_wait(&bars[L::kVFull + j % VS], (j / VS) & 1, abort, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, kv)) {
          if (elected) give_up(p, abort, 9);
          break;
        }
        if (elected) dev::mbar_arrive(&bars[L::kP + 0]);
        if (!__all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kP + 0], j & 1, abort, p.wait_limit_ns))) break;
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs the loop, so its state is warp-uniform; one
      // elected lane issues the MMAs and commits.  Every lane waits, and a
      // vote keeps the warp on one path when a wait gives up.
      const bool leader = dev::elect_one();
      const uint32_t sQ = dev::smem_u32(smem + L::kQ);
      const uint32_t sK = dev::smem_u32(smem + L::kK);
      const uint32_t sV = dev::smem_u32(smem + L::kV);
      constexpr uint32_t idesc_s = dev::idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = dev::idesc_bf16_f32(128, D, false, true);
      // descriptors of the region starts; an operand at byte offset `off`
      // inside a region is its descriptor + off/16 (the address field never
      // carries: shared-memory addresses stay below 2^18)
      const uint64_t dQ = dev::sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK = dev::sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = dev::sdesc_sw128(sV, 16384, 1024);
      auto issue_s = [&](int x, int st) {
        const uint32_t d = tmem + x * 128;
        const uint64_t a0 = dQ + static_cast<uint32_t>(x * (L::kTileBytes >> 4));
        const uint64_t b0 = dK + static_cast<uint32_t>(st * (L::kTileBytes >> 4));
        #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          dev::mma_ss(d, a0 + off, b0 + off, idesc_s, kk > 0);
        }
      };
      // PV over key rows [16*k0, 16*k1) of the tile
      auto issue_pv = [&](int x, int st, bool acc, int k0, int k1) {
        const uint32_t d = tmem + 256 + x * D;
        const uint64_t b0 = dV + static_cast<uint32_t>(st * (L::kTileBytes >> 4));
        #pragma unroll
        for (int kk = k0; kk < k1; ++kk)
          dev::mma_ts(d, tmem + x * 128 + kk * 8, b0 + static_cast<uint32_t>(kk * (2048 >> 4)), idesc_o,
                      (acc || kk > 0) ? 1u : 0u);
      };
      const bool ok = __all_sync(0xffffffffu, dev::mbar_wait(&bars[ROPE_Q ? L::kQReady : L::kQFull], 0, abort, p.wait_limit_ns) &&
                                                  dev::mbar_wait(&bars[L::kKFull], 0, abort, p.wait_limit_ns));
      if (!ok && leader) give_up(p, abort, 3);
      if (ok) {
        dev::tc_fence_after();
        if (leader) {
          issue_s(0, 0);
          dev::mma_commit(&bars[L::kSFull + 0]);
          issue_s(1, 0);
          dev::mma_commit(&bars[L::kSFull + 1]);
          dev::mma_commit(&bars[L::kKEmpty + 0]);
        }
        for (int j = 0; j < n; ++j) {
          const int vst = j % VS;
          const bool more = j + 1 < n;
          const int kst1 = (j + 1) % KS;
          // P of tile 0 also means V(j) and K(j+1) have landed (warp 3)
          if (!__all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kP + 0], j & 1, abort, p.wait_limit_ns))) {
            if (leader) give_up(p, abort, 4);
            break;
          }
          dev::tc_fence_after();
          if (leader) {
            issue_pv(0, vst, j > 0, 0, 8);
            if (more) {
              issue_s(0, kst1);
              dev::mma_commit(&bars[L::kSFull + 0]);
            }
          }
          if (!__all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kP + 1], j & 1, abort, p.wait_limit_ns))) {
            if (leader) give_up(p, abort, 6);
            break;
          }
          dev::tc_fence_after();
          if (leader) {
            issue_pv(1, vst, j > 0, 0, 8);
            dev::mma_commit(&bars[L::kVEmpty + vst]);
            if (more) {
              issue_s(1, kst1);
              dev::mma_commit(&bars[L::kSFull + 1]);
              dev::mma_commit(&bars[L::kKEmpty + kst1]);
            }
          }
        }
        if (leader) {
          dev::mma_commit(&bars[L::kODone + 0]);
          dev::mma_commit(&bars[L::kODone + 1]);
        }
      }
      // drain: all issued MMAs complete before TMEM is released
      if (leader) dev::mma_commit(&bars[L::kDrain]);
      __syncwarp();
      volatile int never = 0;
      dev::mbar_wait(&bars[L::kDrain], 0, &never, p.wait_limit_ns);
    }
  } else {
    dev::setmaxnreg_inc<kRegsHigh>();
    if constexpr (ROPE_Q) {
      // ------------------------------------------------ RoPE of the Q tiles
      // the table arrived with Q; one thread rotates one query row
      const float2* tab = reinterpret_cast<const float2*>(smem + L::kTab);
      const int r = (warp - 4) * 32 + lane;  // 0..255
      const bool qok = __all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kQFull], 0, abort, p.wait_limit_ns));
      if (qok) {
        if (q0 + r < p.n_q) rope_q_row<D>(smem + L::kQ, L::kTileBytes, tab, r, q0, p);
        // the rotated tiles are read by the tensor core (async proxy)
        dev::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&bars[L::kQReady]);
      } else {
        give_up(p, abort, 10);
      }
    }
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + x * 128;
    const uint32_t tO = tmem + lane_off + 256 + x * D;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      int seg, row0, valid;
      tile_of(p, j, seg, row0, valid);
      // every lane polls the barrier; a vote keeps the warp on one path
      ok = __all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kSFull + x], j & 1, abort, p.wait_limit_ns));
      if (!ok) {
        give_up(p, abort, 7);
        break;
      }
      dev::tc_fence_after();
      // Exponentials against the running max m, no row max: if the tile's
      // probabilities sum to at most 2^8, none exceeds 2^8 (the bound the lazy
      // rescale keeps).  Otherwise (always on the first tile, rarely later)
      // the row takes the exact max of the tile, O and l are rescaled, and the
      // tile is recomputed; S is still intact in tensor memory until P is
      // written over it.
      uint32_t pk[64];
      float l0 = 0.f, l1 = 0.f;
      {
        uint32_t sr[128];
        load_scores(tS, sr, valid);
        tile_exp<EXACT_L>(reinterpret_cast<const float*>(sr), sl2, -m, pk, l0, l1);
      }
      const bool need = !(l0 + l1 <= kTileSumLimit);  // also true for inf / NaN (first tile: m = -inf)
      if (__any_sync(0xffffffffu, need)) {
        uint32_t sr[128];
        load_scores(tS, sr, valid);
        const float* s = reinterpret_cast<const float*>(sr);
        const float mx = row_max(s) * sl2;
        const float m_new = fmaxf(m, mx);
        const float alpha = need ? dev::ex2_approx(m - m_new) : 1.f;
        if (need) {
          m = m_new;
          l *= alpha;
        }
        if (j > 0) {
          #pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            dev::tmem_ld32(tO + c, o);
            #pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            dev::tmem_st32(tO + c, o);
          }
        }
        l0 = 0.f;
        l1 = 0.f;
        tile_exp<EXACT_L>(s, sl2, -m, pk, l0, l1);
      }
      {
        uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
        uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
        dev::tmem_st32(tS, p0);
        dev::tmem_st32(tS + 32, p1);
      }
      // publish the tile's probabilities: the PV product may start
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&bars[L::kP + x]);
      l += l0 + l1;
    }
    if (ok) ok = __all_sync(0xffffffffu, dev::mbar_wait(&bars[L::kODone + x], 0, abort, p.wait_limit_ns));
    if (ok) {
      dev::tc_fence_after();
      const int q = q0 + x * 128 + row;
      const float inv_l = 1.f / l;
      // O leaves through shared memory: Q tile x is free (every MMA, and so
      // every read of Q, has completed once O is done).  Each thread writes
      // its row in the same 128-byte-swizzled layout the loads use; then one
      // tensor-map store per 64 columns writes the warp's 32 rows, clipped
      // at n_q.
      uint8_t* sO = smem + L::kQ + x * L::kTileBytes;
      #pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        dev::tmem_ld32(tO + c, o);
        uint32_t pk[16];
        #pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = dev::pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                   __uint_as_float(o[2 * i + 1]) * inv_l);
        uint8_t* rowp = sO + (c >> 6) * 16384 + row * 128;
        const int j0 = (c & 63) >> 3;
        #pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(rowp + (((j0 + i) ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      dev::fence_proxy_async_smem();
      __syncwarp();
      const int wrow0 = q0 + x * 128 + quad * 32;
      if (lane == 0 && wrow0 < p.n_q) {
        #pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          dev::tma_store_4d(&maps.o, sO + cb * 16384 + quad * 32 * 128, cb * 64, h, wrow0, b);
        dev::bulk_commit();
        // the block's shared memory must outlive the reads of the stores
        dev::bulk_wait_read_all();
      }
      if (p.lse != nullptr && q < p.n_q)
        p.lse[(static_cast<int64_t>(b) * p.H + h) * p.n_q + q] =
            (m + log2f(l)) * 0.69314718055994530942f;
    } else {
      give_up(p, abort, 8);
    }
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, 512);
  }
}

int make_token_map(CUtensorMap* m, const void* ptr, int B, int64_t N, int H, int D, uint32_t box_rows = 128) {
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)H, (uint64_t)N, (uint64_t)B};
  const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)H * D * 2, (uint64_t)N * H * D * 2};
  const uint32_t box[4] = {64, 1, box_rows, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// Sets a kernel's shared-memory limit and checks its register count against
// the setmaxnreg split, once per device.
template <typename Kernel>
int prepare_kernel(Kernel kernel, bool* done) {
  int dev_id = 0;
  SAVGB_CUDA(cudaGetDevice(&dev_id));
  if (done[dev_id & 63]) return SAVGB_OK;
  SAVGB_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));
  cudaFuncAttributes fa;
  SAVGB_CUDA(cudaFuncGetAttributes(&fa, kernel));
  if (fa.numRegs * kThreads < kRegPoolNeeded)
    return fail(SAVGB_ERR_UNSUPPORTED,
                "chunk_attention: kernel built with %d registers/thread; its register split needs %d",
                fa.numRegs, (kRegPoolNeeded + kThreads - 1) / kThreads);
  done[dev_id & 63] = true;
  return SAVGB_OK;
}

template <int D, int KS, int VS, bool ROPE_Q>
int launch_impl(const void* q, int B, int64_t n_q, int H, const AttnSeg* segs, int n_segs,
                float scale, void* o, float* lse, const QRope* rope, cudaStream_t stream, bool exact_req) {
  using L = Layout<D, KS, VS>;
  const float default_scale = 1.0f / std::sqrt((float)D);
  if (!(scale > 0.f)) scale = default_scale;
  // fp32 exponentials and exact row sums for the log-sum-exp output, on
  // request, and for logits sharper than the default scale's, where the
  // packed form's bf16-rounded exponents cost the most precision
  const bool exact = lse != nullptr || exact_req || scale > kExactScaleRatio * default_scale;
  static bool ready[2][64] = {};
  auto kernel = exact ? attn_fwd_kernel<D, KS, VS, ROPE_Q, true> : attn_fwd_kernel<D, KS, VS, ROPE_Q, false>;
  int rc = prepare_kernel(kernel, ready[exact ? 1 : 0]);
  if (rc) return rc;
  AttnMaps maps;
  if ((rc = make_token_map(&maps.q, q, B, n_q, H, D))) return rc;
  if ((rc = make_token_map(&maps.o, o, B, n_q, H, D, 32))) return rc;
  AttnParams p{};
  p.n_q = (int)n_q;
  p.H = H;
  p.n_tiles = 0;
  for (int s = 0; s < 3; ++s) {
    const bool used = s < n_segs && segs[s].n > 0;
    p.seg_len[s] = used ? (int)segs[s].n : 0;
    p.seg_tiles[s] = used ? (int)((segs[s].n + kTileKV - 1) / kTileKV) : 0;
    p.n_tiles += p.seg_tiles[s];
    if (used) {
      if ((rc = make_token_map(&maps.k[s], segs[s].k, B, segs[s].n, H, D))) return rc;
      if ((rc = make_token_map(&maps.v[s], segs[s].v, B, segs[s].n, H, D))) return rc;
    } else {
      maps.k[s] = maps.q;
      maps.v[s] = maps.q;
    }
  }
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse = lse;
  int dyn_smem = L::kDynSmem;
  if (rope) {
    using R = RopeSplit<D>;
    p.gh = rope->grid_h;
    p.gw = rope->grid_w;
    p.t0 = rope->t0;
    p.rope_tab = static_cast<const float2*>(rope->tab);
    p.tab_t_lo = rope->tab_t_lo;
    p.tab_t_n = rope->tab_t_n;
    const int64_t hw = (int64_t)rope->grid_h * rope->grid_w;
    p.tab_t_rows = (int)std::min<int64_t>((kBlockQ - 1) / hw + 2, rope->tab_t_n);
    p.tab_h_sec = (int)even_up((int64_t)p.gh * R::kH);
    p.tab_hw_entries = p.tab_h_sec + (int)even_up((int64_t)p.gw * R::kW);
    const int64_t tab = 8 * ((int64_t)p.tab_t_rows * R::kT + p.tab_hw_entries);
    if (L::kTab + tab + 1024 > 227 * 1024)
      return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention_qrope: RoPE tables of %lld bytes do not fit", (long long)tab);
    dyn_smem = std::max<int>(dyn_smem, L::kTab + 1024 + (int)tab);
  }
  if ((rc = error_word(&p.err))) return rc;
  p.fault_tile = -1;
  p.wait_limit_ns = dev::kWaitLimitNs;
  ArmedFault fault;
  if (take_fault(SAVGB_FAULT_ATTENTION_K_TILE, &fault)) {
    p.fault_tile = fault.index;
    p.wait_limit_ns = fault.limit_ns;
  }
  dim3 grid((unsigned)((n_q + kBlockQ - 1) / kBlockQ), (unsigned)H, (unsigned)B);
  SAVGB_CUDA(launch_dependent(kernel, grid, dim3(kThreads), dyn_smem, stream, maps, p));
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

}  // namespace

int validate_attention(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                       int n_segs, const void* o) {
  if (!q || !o) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: null q or o");
  if (!aligned16(q) || !aligned16(o)) return fail(SAVGB_ERR_ALIGNMENT, "chunk_attention: q and o must be 16-byte aligned");
  if (D != 64 && D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention: head_dim %d (64 or 128 supported)", D);
  if (B < 1 || B > 65535 || H < 1 || H > 65535) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: B and H must be in [1, 65535]");
  if (n_q < 1 || n_q > (int64_t)1 << 30) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: n_q must be in [1, 2^30]");
  if (n_segs < 1 || n_segs > 3 || !segs) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: 1 to 3 segments");
  int64_t total = 0;
  for (int s = 0; s < n_segs; ++s) {
    if (segs[s].n < 0 || segs[s].n > (int64_t)1 << 30) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: segment %d size", s);
    if (segs[s].n == 0) continue;
    if (!segs[s].k || !segs[s].v) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: segment %d has null k or v", s);
    if (!aligned16(segs[s].k) || !aligned16(segs[s].v)) return fail(SAVGB_ERR_ALIGNMENT, "chunk_attention: segment %d not 16-byte aligned", s);
    total += segs[s].n;
  }
  if (total < 1) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention: no key/value tokens");
  return SAVGB_OK;
}

int launch_attention(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                     int n_segs, float scale, void* o, float* lse, cudaStream_t stream, bool exact_softmax) {
  int rc = check_device(nullptr);
  if (rc) return rc;
  if (D == 64)
    return launch_impl<64, kStagesK64, kStagesV64, false>(q, B, n_q, H, segs, n_segs, scale, o, lse, nullptr, stream,
                                                          exact_softmax);
  return launch_impl<128, kStagesK128, kStagesV128, false>(q, B, n_q, H, segs, n_segs, scale, o, lse, nullptr,
                                                          stream, exact_softmax);
}

int validate_qrope(const QRope& r, int64_t n_q, int D) {
  if (r.grid_t < 1 || r.grid_h < 1 || r.grid_w < 1 || r.grid_h > 4096 || r.grid_w > 4096)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope: grid sizes must be >= 1 (h, w <= 4096)");
  if ((int64_t)r.grid_t * r.grid_h * r.grid_w != n_q)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope: n_q != grid_t*grid_h*grid_w");
  if (!(r.base > 0.0) || !std::isfinite(r.base))
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope: base must be finite and > 0");
  if (r.t0 < -(1 << 20) || r.t0 > (1 << 20)) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope: |t0| > 2^20");
  if (D != 64 && D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention_qrope: head_dim %d", D);
  if (r.tab && (!aligned16(r.tab) || r.t0 < r.tab_t_lo || (int64_t)r.t0 + r.grid_t > (int64_t)r.tab_t_lo + r.tab_t_n))
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope: the RoPE table does not cover the query frames");
  return SAVGB_OK;
}

namespace {

template <int D>
int64_t table_entries(int n_t, int grid_h, int grid_w) {
  using R = RopeSplit<D>;
  return even_up((int64_t)n_t * R::kT) + even_up((int64_t)grid_h * R::kH) + even_up((int64_t)grid_w * R::kW);
}

template <int D, int KS, int VS>
bool fits(int grid_t, int grid_h, int grid_w) {
  using R = RopeSplit<D>;
  using L = Layout<D, KS, VS>;
  const int64_t hw = (int64_t)grid_h * grid_w;
  const int64_t rows = std::min<int64_t>((kBlockQ - 1) / hw + 2, grid_t);
  const int64_t tab = 8 * (rows * R::kT + even_up((int64_t)grid_h * R::kH) + even_up((int64_t)grid_w * R::kW));
  return L::kTab + tab + 1024 <= 227 * 1024;
}

}  // namespace

int64_t rope_q_table_bytes(int D, int n_t, int grid_h, int grid_w) {
  return 8 * (D == 64 ? table_entries<64>(n_t, grid_h, grid_w) : table_entries<128>(n_t, grid_h, grid_w));
}

bool qrope_fits(int D, int grid_t, int grid_h, int grid_w) {
  if (D == 64) return fits<64, kStagesK64, kStagesV64>(grid_t, grid_h, grid_w);
  if (D == 128) return fits<128, 2, kStagesV128>(grid_t, grid_h, grid_w);
  return false;
}

int rope_q_table_build(void* tab, int D, int t_lo, int n_t, int grid_h, int grid_w, double base,
                       cudaStream_t stream) {
  const int64_t entries = rope_q_table_bytes(D, n_t, grid_h, grid_w) / 8;
  const int threads = 256;
  const int blocks = (int)std::min<int64_t>((entries + threads - 1) / threads, 1024);
  const float log2_base = (float)std::log2(base);
  // an ordinary launch: it starts after everything before it on the stream
  if (D == 64)
    rope_q_table_kernel<64><<<blocks, threads, 0, stream>>>(static_cast<float2*>(tab), t_lo, n_t, grid_h, grid_w,
                                                             log2_base);
  else
    rope_q_table_kernel<128><<<blocks, threads, 0, stream>>>(static_cast<float2*>(tab), t_lo, n_t, grid_h, grid_w,
                                                              log2_base);
  SAVGB_CUDA(cudaGetLastError());
  note_launch();
  return SAVGB_OK;
}

int launch_attention_qrope(const void* q, int B, int64_t n_q, int H, int D, const AttnSeg* segs,
                           int n_segs, float scale, const QRope& rope, void* o, float* lse,
                           cudaStream_t stream, bool exact_softmax) {
  int rc = check_device(nullptr);
  if (rc) return rc;
  if (!qrope_fits(D, rope.tab ? rope.tab_t_n : rope.grid_t, rope.grid_h, rope.grid_w))
    return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention_qrope: the RoPE tables of a %d x %d grid do not fit in "
                "shared memory", rope.grid_h, rope.grid_w);
  QRope r = rope;
  void* tmp = nullptr;
  if (!r.tab) {
    // a table for this call only, stream-ordered
    SAVGB_CUDA(cudaMallocAsync(&tmp, (size_t)rope_q_table_bytes(D, r.grid_t, r.grid_h, r.grid_w), stream));
    rc = rope_q_table_build(tmp, D, r.t0, r.grid_t, r.grid_h, r.grid_w, r.base, stream);
    r.tab = tmp;
    r.tab_t_lo = r.t0;
    r.tab_t_n = r.grid_t;
  }
  if (!rc) {
    if (D == 64)
      rc = launch_impl<64, kStagesK64, kStagesV64, true>(q, B, n_q, H, segs, n_segs, scale, o, lse, &r, stream,
                                                         exact_softmax);
    else  // two K stages leave room for the tables (and run as fast as three)
      rc = launch_impl<128, 2, kStagesV128, true>(q, B, n_q, H, segs, n_segs, scale, o, lse, &r, stream,
                                                  exact_softmax);
  }
  if (tmp) {
    const cudaError_t e = cudaFreeAsync(tmp, stream);
    if (!rc && e != cudaSuccess) rc = cuda_fail(e, "cudaFreeAsync(RoPE table)");
  }
  return rc;
}

}  // namespace savgb

extern "C" int chunk_attention(const void* q, int B, int64_t n_q, int H, int D,
                               const savgb_kv_segment* segs, int n_segs, float scale, void* o,
                               float* lse, void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:chunk_attention");
  clear_error();
  AttnSeg s[3] = {};
  if (segs && n_segs >= 1 && n_segs <= 3)
    for (int i = 0; i < n_segs; ++i) s[i] = AttnSeg{segs[i].k, segs[i].v, segs[i].n_tokens};
  int rc = validate_attention(q, B, n_q, H, D, segs ? s : nullptr, n_segs, o);
  if (rc) return rc;
  return launch_attention(q, B, n_q, H, D, s, n_segs, scale, o, lse,
                          static_cast<cudaStream_t>(stream));
}

extern "C" int chunk_attention_qrope(const void* q, int B, int64_t n_q, int H, int D, int grid_t, int grid_h,
                                     int grid_w, int t0, double base, const savgb_kv_segment* segs, int n_segs,
                                     float scale, void* o, float* lse, void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:chunk_attention_qrope");
  clear_error();
  AttnSeg sg[3] = {};
  if (segs && n_segs >= 1 && n_segs <= 3)
    for (int i = 0; i < n_segs; ++i) sg[i] = AttnSeg{segs[i].k, segs[i].v, segs[i].n_tokens};
  int rc = validate_attention(q, B, n_q, H, D, segs ? sg : nullptr, n_segs, o);
  if (rc) return rc;
  const QRope r{grid_t, grid_h, grid_w, t0, base};
  if ((rc = validate_qrope(r, n_q, D))) return rc;
  return launch_attention_qrope(q, B, n_q, H, D, sg, n_segs, scale, r, o, lse, static_cast<cudaStream_t>(stream));
}

extern "C" int chunk_attention_qrope_fits(int D, int grid_t, int grid_h, int grid_w, int* fits) {
  using namespace savgb;
  clear_error();
  if (!fits) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_fits: null output");
  *fits = 0;
  if (grid_t < 1 || grid_h < 1 || grid_w < 1)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_fits: grid sizes must be >= 1");
  *fits = (grid_h <= 4096 && grid_w <= 4096 && qrope_fits(D, grid_t, grid_h, grid_w)) ? 1 : 0;
  return SAVGB_OK;
}

extern "C" int chunk_attention_qrope_table_bytes(int D, int grid_t, int grid_h, int grid_w, int64_t* bytes) {
  using namespace savgb;
  clear_error();
  if (!bytes) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_table_bytes: null output");
  *bytes = 0;
  if (D != 64 && D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention_qrope_table_bytes: head_dim %d", D);
  if (grid_t < 1 || grid_h < 1 || grid_w < 1 || grid_t > 4096 || grid_h > 4096 || grid_w > 4096)
    return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_table_bytes: grid sizes must be in [1, 4096]");
  *bytes = rope_q_table_bytes(D, grid_t, grid_h, grid_w);
  return SAVGB_OK;
}

extern "C" int chunk_attention_qrope_build_table(void* table, int D, int grid_t, int grid_h, int grid_w, int t0,
                                                 double base, void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:chunk_attention_qrope_build_table");
  clear_error();
  if (!table) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_build_table: null table");
  if (!aligned16(table)) return fail(SAVGB_ERR_ALIGNMENT, "chunk_attention_qrope_build_table: table not 16-byte aligned");
  if (D != 64 && D != 128) return fail(SAVGB_ERR_UNSUPPORTED, "chunk_attention_qrope_build_table: head_dim %d", D);
  const QRope r{grid_t, grid_h, grid_w, t0, base};
  int rc = validate_qrope(r, (int64_t)grid_t * grid_h * grid_w, D);
  if (rc) return rc;
  if (grid_t > 4096) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_build_table: grid_t > 4096");
  if ((rc = check_device(nullptr))) return rc;
  return rope_q_table_build(table, D, t0, grid_t, grid_h, grid_w, base, static_cast<cudaStream_t>(stream));
}

extern "C" int chunk_attention_qrope_with_table(const void* q, int B, int64_t n_q, int H, int D, int grid_t,
                                                int grid_h, int grid_w, int t0, const void* table,
                                                const savgb_kv_segment* segs, int n_segs, float scale, void* o,
                                                float* lse, void* stream) {
  using namespace savgb;
  savgb::ApiRange api_range_("savgb:chunk_attention_qrope_with_table");
  clear_error();
  if (!table) return fail(SAVGB_ERR_INVALID_ARG, "chunk_attention_qrope_with_table: null table");
  AttnSeg sg[3] = {};
  if (segs && n_segs >= 1 && n_segs <= 3)
    for (int i = 0; i < n_segs; ++i) sg[i] = AttnSeg{segs[i].k, segs[i].v, segs[i].n_tokens};
  int rc = validate_attention(q, B, n_q, H, D, segs ? sg : nullptr, n_segs, o);
  if (rc) return rc;
  // the table holds the angles, so the base only has to pass validation here
  QRope r{grid_t, grid_h, grid_w, t0, 1.0};
  r.tab = table;
  r.tab_t_lo = t0;
  r.tab_t_n = grid_t;
  if ((rc = validate_qrope(r, n_q, D))) return rc;
  return launch_attention_qrope(q, B, n_q, H, D, sg, n_segs, scale, r, o, lse, static_cast<cudaStream_t>(stream));
}
