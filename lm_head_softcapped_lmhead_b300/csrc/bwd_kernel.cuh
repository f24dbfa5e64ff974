// bwd_kernel.cuh -- backward of the fused tied-LM-head + softcapped CE:
//   G_ij = (p_ij - [j == t_i]) (1 - tanh^2(z_ij / c)),  p_ij = e^{s_ij - lse_i}
//   dh = w G W            (rows stationary, "DH" mode)
//   dW (+)= w G^T h       (vocab stationary, "DW" mode)
//   forward + dh in one pass ("FD" mode, below)
// Chain rule of nll_i = lse_i - s_{i,t_i} through s = c tanh(z/c), for the
// training step of "parameter-golf: ... Where Model Size Becomes the Game",
// section "The Baseline Is a Map, Not the Destination" (loss.backward()).
//
// A [128 rows x 512] fp32 accumulator fills all of an SM's TMEM, so the logit
// tile and the accumulator cannot share one SM.  Each stationary block is
// therefore handled by a cluster of two CTAs:
//  * rank 0, the Z CTA: keeps the stationary operand X (128 x d bf16) in
//    TMEM (copied there from the ring with tcgen05.cp), streams the other
//    operand Y in 128-row tiles through a ring of 64 KB TMA loads, computes
//    z = X Y^T (tcgen05, A from TMEM, M=128 N=128, double-buffered in TMEM),
//    and its 16 epilogue warps (one 32-column chunk each per tile) turn each
//    z tile into the bf16 tile P = -G (DH) or -G^T (DW) in the 128B-swizzled
//    K-major layout the A CTA's MMA reads, into a local staging copy; a
//    forwarder warp sends each staged tile to the peer CTA's shared memory
//    (DSMEM) in two bulk copies.
//  * rank 1, the A CTA: loads the same Y tile in 64-row slabs (as the
//    MN-major B operand) and accumulates acc (128 x d fp32, all 512 TMEM
//    columns) += P Y with tcgen05 M=128 N=d/2; after the last tile its 16
//    drain warps scale by w and write dh (bf16) or dW (fp32, added or
//    stored; or a partial for a later ordered reduction when the rows are
//    split across several clusters).
// The logits and G never leave the two SMs.  Every wait is bounded.
//
// FD mode computes the forward (nll, lse) and dh in the same pass over the
// vocabulary, without the forward's lse.  dh_i = w sum_j G_ij W_j splits as
//   dh_i = w [ sum_{j != t_i} p_ij (1 - tanh_ij^2) W_j
//              + (p_{i,t_i} - 1)(1 - tanh_{i,t_i}^2) W_{t_i} ],
// and p_ij = e^{s_ij} / S_i with S_i = sum_j e^{s_ij} constant along the row.
// So the Z CTA streams the unnormalised tile P = e^{s} (tanh^2 - 1) with the
// target column left out (so no large p_t - 1 cancellation happens in bf16),
// and keeps per row S_other = the sum of e^{s} over the non-target columns,
// and the target's e^{s_t} and 1 - tanh^2.  At the end of the row block the
// A CTA's drain forms S = S_other + e^{s_t}, lse = ln S,
// nll = log1p(S_other / e^{s_t}) and dh_i = alpha_i acc_i + beta_i W_{t_i}
// with alpha_i = -w / S and beta_i = -w (S_other / S)(1 - tanh_t^2): no
// quantity there cancels as p_t -> 1.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <string>

#include "ce_math.cuh"
#include "ptx.cuh"
#include "softcap_math.cuh"

namespace lmce {
int make_map_bf16_3d(CUtensorMap* m, const void* base, uint64_t d, uint64_t rows, uint64_t pitch_bytes,
                     uint32_t box_rows, uint32_t box_chunks);
void set_last_error(const std::string& s);
void count_launches(unsigned n);

namespace bwdk {

enum Mode : int { DH = 0, DW = 1, FD = 2 };

constexpr int BM = 128;   // stationary block (TMEM lanes)
constexpr int BT = 128;   // streamed tile (z columns; K of the accumulation)
constexpr int KB = 64;    // K elements per chunk
constexpr int MAX_KC = 8; // d <= 512
constexpr int ZSC = 4;      // chunks per Z ring stage (64 KB, one TMA load)
constexpr int EPI_WARPS = 16;  // Z: epilogue warps; A: drain warps
constexpr int TMA_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int FWD_WARP = 18;   // Z: forwards P tiles to the A CTA; A: acknowledges their arrival
constexpr int THREADS = 608;
constexpr uint32_t CHUNK = 128 * KB * 2;  // 16 KB: 128 rows x 64 bf16
constexpr uint32_t ZSTAGE = ZSC * CHUNK;   // 64 KB
// The A CTA loads its Y tile in 2 slabs of 64 rows x d (one TMA load per
// slab, up to 64 KB); inside a slab the d / 64 chunks of 64 x 64 follow each
// other (8 KB apart).
constexpr int SLAB_ROWS = 64;
constexpr int NSLAB = BT / SLAB_ROWS;
constexpr uint32_t SLAB_CHUNK = SLAB_ROWS * KB * 2;  // 8 KB
constexpr uint32_t P_SLOT = 2 * CHUNK;                // 32 KB: one 128 x 128 bf16 P tile
constexpr uint32_t Z_TMEM_X = 256;  // Z: the stationary block X in TMEM columns 256-511
// FD: per-row records of the Z epilogue, [column group][row] x 32 bytes:
// {float sum of e^s over the non-target columns, unused, float e^{s_t},
//  1 - tanh_t^2, int target, int flags, 2 x unused}.  They go through global memory
// (L2): [cluster][column group][row], so the Z CTA's shared memory holds a
// third P staging copy instead.
constexpr uint32_t REC_BYTES = 32;
constexpr int NREC_GROUPS = EPI_WARPS / 4;
constexpr int kFdRecClusters = 128;  // clusters with a record area (launches use at most this many)
constexpr size_t kFdRecClusterBytes = static_cast<size_t>(NREC_GROUPS) * BM * REC_BYTES;  // 16 KB
constexpr int FL_LIVE = 1, FL_TVALID = 2, FL_HIT = 4;

// Shared-memory plan of a mode.  The Z CTA holds a ring of Y stages (X is in
// TMEM) and the P staging copies; the A CTA holds a ring of Y slabs and the P
// slots.  The Z epilogue writes each P tile into a local staging copy, and
// the forwarder warp sends each 16 KB column chunk of it with one bulk DSMEM
// copy into an A CTA P slot.
// What the measurements favoured (N=65536, V=8192, d=512, ms per pass): few
// large transfers between the CTAs' rings over many small ones.  Y slabs of
// 64 rows (two 64 KB slots) against 32 rows (two 32 KB slots, 4-5 P slots):
// DW 0.983 against 1.078, DH 0.936 against 0.954, FD 1.018 against 1.044
// (the 32-row FD form stored P into the peer with st.async, which was the
// faster hand-off there); four 16-row slots in the same 64 KB made every pass
// 40 % slower, and four 32-row slots in 128 KB were slower than two 64-row
// ones (DW 1.135 against 1.004).  One 32 KB bulk copy per tile instead of
// two 16 KB copies: FD 1.021, DW 0.991.  Three staging copies against two:
// DW 0.983 against 1.004, FD 0.973 against 1.016 (FD's row records moved to
// global memory to make room).
template <int MODE>
struct Cfg {
  static constexpr int YSTAGES = 2;               // Z ring stages (64 KB)
  static constexpr int NSTG = 3;                  // Z: P staging copies (32 KB)
  static constexpr int ASLOTS = 2;                // A: Y slab slots (64 KB)
  static constexpr int NPS = 3;                   // A: P slots (32 KB)
  // Z CTA layout
  static constexpr uint32_t Z_Y = 0;
  static constexpr uint32_t Z_STG = Z_Y + YSTAGES * ZSTAGE;          // NSTG x 2 x 16 KB
  static constexpr uint32_t Z_END = Z_STG + NSTG * 2 * CHUNK;
  // A CTA layout
  static constexpr uint32_t A_Y = 0;
  static constexpr uint32_t A_P = A_Y + ASLOTS * MAX_KC * SLAB_CHUNK;
  static constexpr uint32_t A_END = A_P + NPS * P_SLOT;
  static constexpr uint32_t BAR_OFF = (Z_END > A_END ? Z_END : A_END);
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 512 + 1024;
  // mbarrier indices (8 bytes each) from BAR_OFF; bytes 504..511 hold the
  // TMEM address and the abort flag.
  static constexpr int B_ZY_FULL = 0;                      // [YSTAGES]
  static constexpr int B_ZY_EMPTY = B_ZY_FULL + YSTAGES;   // [YSTAGES]
  static constexpr int B_X_FREE = B_ZY_EMPTY + YSTAGES;
  static constexpr int B_X_READY = B_X_FREE + 1;
  static constexpr int B_ACC_FULL = B_X_READY + 1;         // [2]
  static constexpr int B_ACC_EMPTY = B_ACC_FULL + 2;       // [2]
  static constexpr int B_P_EMPTY = B_ACC_EMPTY + 2;        // [NPS]
  static constexpr int B_P_FULL = B_P_EMPTY + NPS;         // [NPS]
  static constexpr int B_AY_FULL = B_P_FULL + NPS;         // [ASLOTS]
  static constexpr int B_AY_EMPTY = B_AY_FULL + ASLOTS;    // [ASLOTS]
  static constexpr int B_MMA_DONE = B_AY_EMPTY + ASLOTS;
  static constexpr int B_RD_FULL = B_MMA_DONE + 1;
  static constexpr int B_RD_EMPTY = B_RD_FULL + 1;
  static constexpr int B_STG_FULL = B_RD_EMPTY + 1;        // [NSTG][2]
  static constexpr int B_STG_EMPTY = B_STG_FULL + 2 * NSTG;  // [NSTG]
  static_assert((B_STG_EMPTY + NSTG) * 8 <= 504, "mbarriers overlap the TMEM address slot");
  static_assert(SMEM_BYTES <= 232448, "shared memory above the 227 KB per-CTA limit");
};
constexpr uint32_t Z_TMEM_COLS = 512;
constexpr uint32_t A_TMEM_COLS = 512;
constexpr uint32_t IDESC_Z = idesc_bf16_f32(128, BT, false, false);
constexpr int MAX_SPLIT = 8;

struct Params {
  int N, V, d, KC;
  int n_tiles;          // streamed tiles per stationary block (whole range)
  int n_blocks;         // stationary blocks
  int split;            // DW: row splits per vocab block (1 = direct output)
  int n_units;          // n_blocks * split
  const int64_t* tgt;   // [N]
  const uint8_t* mask;  // [N] or null
  const float* lse;     // [N]
  const float* nll_in;  // [N] from the same forward, or null: the target's p - 1 = expm1(-nll)
  float inv_c, cl2e, w;  // w: the drain's scale (-grad_scale: the tiles hold -G; FD: +grad_scale)
  float c;
  const __nv_bfloat16* W;  // FD: the head, for the target-row term of dh
  float* nll;              // FD outputs [N]
  float* lse_out;
  __nv_bfloat16* dh;    // DH output [N, ldh]
  long long ldh;
  float* dW;            // DW output [V, d]
  int accumulate;
  float* dw_part;       // DW split partials [split][V_pad][d]
  int V_pad;
  uint4* fd_rec;        // FD row records [cluster][NREC_GROUPS][BM] x 2 uint4 (global memory)
  unsigned* status;
  float xlim;           // DH, DW: kTanhXmax, or +inf with no cap (the SFU tanh's range)
};

// The epilogue forms the NEGATED gradient tile, P = -G (or -G^T), because
// then exponent and derivative are one FFMA2 each:
//   a = cl2e * tanh - lse2,  p = 2^a,
//   w = tanh^2 - 1 = -(1 - tanh^2),
//   -G = (p - [j == t]) * w.
// The drain multiplies the accumulator by -grad_scale.
// tanh(z/c) comes from the SFU (tanh.approx.f32) for chunks with every
// |z| / c <= kTanhXmax; the others take the exact form out of line.  Over
// that range its relative error measured at most 9.9e-6 (every float in
// [1e-6, 0.3] on a B300; mean signed error at most 2.2e-6 in any decade),
// which puts at most 8e-5 on s at c = 30 and about 5e-6 at the logits of a
// 0.02-scale head: far below the bf16 rounding of the gradient tile, and
// below the forward's tolerance in FD's row sums (nll and lse).  The FMA
// pipe, which slows the Z CTA's tensor pipe when busy, then carries 4 (DH,
// DW) or 5 (FD) packed operations per logit pair instead of 7 or 8 with the
// degree-2 polynomial; at N = 65536 the FD pass went 0.963 -> 0.905 ms, dW
// 0.983 -> 0.946 ms and dh 0.936 -> 0.875 ms.
struct EpiConst {
  float2 cl2e2;   // c log2(e)
  float2 invc2;   // 1 / c
  float2 m1;      // -1
  float xlim;     // kTanhXmax (|z| / c above it takes the exact slow path)
  float inv_c, cl2e;
};


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Slow path for chunks whose |z| may exceed the polynomial range: exact-form
// tanh per element, same sign convention.  Kept out of line (arguments and
// result by value) so the compiler branches to it instead of predicating it
// into every chunk; only the call site copies the chunk to the stack.
struct Chunk32 {
  uint32_t v[32];
};
struct Packed16 {
  uint32_t v[16];
};
// At the target column p - 1 is either formed here (pp - 1) or, when the
// forward's nll is known (use_pm1), taken as expm1(-nll): that keeps its
// relative precision when p_t -> 1, where s_t - lse cancels in fp32.
// DH: one row per thread (lse2_row, target column rel, valid columns lim).
__device__ __noinline__ Packed16 g_chunk_slow_dh(Chunk32 r, float inv_c, float cl2e, float lse2_row, int rel, int lim,
                                                 int use_pm1, float pm1_row) {
  Packed16 out;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float g[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float th = tanh_any(__uint_as_float(r.v[j + e]) * inv_c);
      float pp = ex2_approx(fmaf(th, cl2e, -lse2_row));
      if (j + e == rel) pp = use_pm1 ? pm1_row : pp - 1.0f;
      g[e] = (j + e < lim) ? pp * fmaf(th, th, -1.0f) : 0.f;
    }
    out.v[j / 2] = pack_bf16x2(g[0], g[1]);
  }
  return out;
}
// DW: lane = vocab row, column j = tile row j; lane j holds column j's
// -lse log2(e) (nl_col), target lane (hit_col) and p_t - 1 (pm1_col), read
// by every lane with shuffles (the whole warp calls this).
__device__ __noinline__ Packed16 g_chunk_slow_dw(Chunk32 r, float inv_c, float cl2e, float nl_col, int hit_col,
                                                 float pm1_col, int my_lane, int use_pm1) {
  Packed16 out;
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float g[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float th = tanh_any(__uint_as_float(r.v[j + e]) * inv_c);
      const float nl = __shfl_sync(0xffffffffu, nl_col, j + e);
      const int hit = __shfl_sync(0xffffffffu, hit_col, j + e);
      const float q1 = __shfl_sync(0xffffffffu, pm1_col, j + e);
      float pp = ex2_approx(fmaf(th, cl2e, nl));
      if (hit == my_lane) pp = use_pm1 ? q1 : pp - 1.0f;
      g[e] = pp * fmaf(th, th, -1.0f);
    }
    out.v[j / 2] = pack_bf16x2(g[0], g[1]);
  }
  return out;
}

// DH mode: 32 vocab columns of this thread's row (lse2 = lse log2 e of the
// row, rel = target column inside the chunk or -1, lim = valid columns).
template <bool kHit>
__device__ __forceinline__ void g_chunk_dh(const uint32_t (&r)[32], const EpiConst& k, float lse2, int rel, int lim,
                                           int use_pm1, float pm1, uint32_t (&out)[16]) {
  const float2 nl = make_float2(-lse2, -lse2);
  float mu = 0.f;  // max |z| / c of the chunk (range of the fast path)
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 z = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    const float2 x = __fmul2_rn(z, k.invc2);
    mu = fmax3(mu, fabsf(x.x), fabsf(x.y));
    const float2 th = make_float2(tanh_sfu(x.x), tanh_sfu(x.y));
    const float2 a = __ffma2_rn(th, k.cl2e2, nl);
    float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    if (kHit) {
      if (2 * j == rel) pp.x = use_pm1 ? pm1 : pp.x - 1.0f;
      if (2 * j + 1 == rel) pp.y = use_pm1 ? pm1 : pp.y - 1.0f;
    }
    float2 g = __fmul2_rn(pp, __ffma2_rn(th, th, k.m1));
    if (lim < 32) {
      g.x = (2 * j < lim) ? g.x : 0.f;
      g.y = (2 * j + 1 < lim) ? g.y : 0.f;
    }
    out[j] = pack_bf16x2(g.x, g.y);
  }
  if (__any_sync(0xffffffffu, !(mu <= k.xlim))) {
    Chunk32 c;
#pragma unroll
    for (int j = 0; j < 32; ++j) c.v[j] = r[j];
    const Packed16 o = g_chunk_slow_dh(c, k.inv_c, k.cl2e, lse2, rel, lim, use_pm1, pm1);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = o.v[j];
  }
}

// DW mode: lane = vocab row of the block, 32 columns = rows of the tile.
// Lane j holds, for column j of the chunk, -lse log2(e) (nl_col, -inf for rows
// that do not count) and the block lane of that row's target (hit_col, -1 if
// outside the block); every lane reads them with shuffles.
template <bool kHit>
__device__ __forceinline__ void g_chunk_dw(const uint32_t (&r)[32], const EpiConst& k, float nl_col, int hit_col,
                                           int my_lane, int use_pm1, float pm1_col, uint32_t (&out)[16]) {
  float mu = 0.f;  // max |z| / c of the chunk (range of the fast path)
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 z = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    const float2 x = __fmul2_rn(z, k.invc2);
    mu = fmax3(mu, fabsf(x.x), fabsf(x.y));
    const float2 th = make_float2(tanh_sfu(x.x), tanh_sfu(x.y));
    const float2 nl = make_float2(__shfl_sync(0xffffffffu, nl_col, 2 * j), __shfl_sync(0xffffffffu, nl_col, 2 * j + 1));
    const float2 a = __ffma2_rn(th, k.cl2e2, nl);
    float2 pp = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    if (kHit) {
      const float qx = __shfl_sync(0xffffffffu, pm1_col, 2 * j);
      const float qy = __shfl_sync(0xffffffffu, pm1_col, 2 * j + 1);
      if (__shfl_sync(0xffffffffu, hit_col, 2 * j) == my_lane) pp.x = use_pm1 ? qx : pp.x - 1.0f;
      if (__shfl_sync(0xffffffffu, hit_col, 2 * j + 1) == my_lane) pp.y = use_pm1 ? qy : pp.y - 1.0f;
    }
    const float2 g = __fmul2_rn(pp, __ffma2_rn(th, th, k.m1));
    out[j] = pack_bf16x2(g.x, g.y);
  }
  if (__any_sync(0xffffffffu, !(mu <= k.xlim))) {
    Chunk32 c;
#pragma unroll
    for (int j = 0; j < 32; ++j) c.v[j] = r[j];
    const Packed16 o = g_chunk_slow_dw(c, k.inv_c, k.cl2e, nl_col, hit_col, pm1_col, my_lane, use_pm1);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = o.v[j];
  }
}

// FD mode: 32 vocab columns of this thread's row.  e = e^{s} =
// 2^(c log2(e) tanh + nl) (nl = 0, or -inf for a row that does not count;
// 0 past column lim), P = e (tanh^2 - 1) except at the target column (rel),
// where P = 0 and e, 1 - tanh^2 go to tg.  Returns the chunk's sum of e over
// its non-target columns.
struct FdTarget {
  float e, om;
};
struct FdSlowOut {
  uint32_t v[16];
  float sum;
  FdTarget tg;
};
__device__ __noinline__ FdSlowOut fd_chunk_slow(Chunk32 r, float inv_c, float cl2e, float nl, int rel, int lim) {
  FdSlowOut o;
  o.sum = 0.f;
  o.tg = FdTarget{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float g[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float z = __uint_as_float(r.v[j + e]);
      const float th = tanh_any(z * inv_c);
      const float ee = (j + e < lim) ? ex2_approx(fmaf(th, cl2e, nl)) : 0.f;
      const float om = fmaf(-th, th, 1.0f);
      float gg = -ee * om;
      if (j + e == rel) {
        o.tg = FdTarget{ee, om};
        gg = 0.f;
      } else {
        o.sum += ee;
      }
      g[e] = gg;
    }
    o.v[j / 2] = pack_bf16x2(g[0], g[1]);
  }
  return o;
}
template <bool kHit>
__device__ __forceinline__ float g_chunk_fd(const uint32_t (&r)[32], const EpiConst& k, float nl, int rel, int lim,
                                            uint32_t (&out)[16], FdTarget& tg) {
  const float2 nl2 = make_float2(nl, nl);
  float mu = 0.f;  // max |z| / c of the chunk (range of the fast path)
  float2 se = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float2 z = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
    const float2 x = __fmul2_rn(z, k.invc2);
    mu = fmax3(mu, fabsf(x.x), fabsf(x.y));
    const float2 th = make_float2(tanh_sfu(x.x), tanh_sfu(x.y));
    const float2 a = __ffma2_rn(th, k.cl2e2, nl2);
    float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
    if (lim < 32) {
      e.x = (2 * j < lim) ? e.x : 0.f;
      e.y = (2 * j + 1 < lim) ? e.y : 0.f;
    }
    const float2 w = __ffma2_rn(th, th, k.m1);
    if (kHit) {
      if (2 * j == rel) {
        tg = FdTarget{e.x, -w.x};
        e.x = 0.f;
      }
      if (2 * j + 1 == rel) {
        tg = FdTarget{e.y, -w.y};
        e.y = 0.f;
      }
    }
    se = __fadd2_rn(se, e);
    const float2 g = __fmul2_rn(e, w);
    out[j] = pack_bf16x2(g.x, g.y);
  }
  float sum = se.x + se.y;
  if (__any_sync(0xffffffffu, !(mu <= k.xlim))) {
    Chunk32 c;
#pragma unroll
    for (int j = 0; j < 32; ++j) c.v[j] = r[j];
    const FdSlowOut o = fd_chunk_slow(c, k.inv_c, k.cl2e, nl, rel, lim);
#pragma unroll
    for (int j = 0; j < 16; ++j) out[j] = o.v[j];
    sum = o.sum;
    if (kHit) tg = o.tg;
  }
  return sum;
}

// A unit's tiles are visited from an offset that depends on its cluster
// slot: clusters that swept the streamed operand in the same order would all
// request the same tile from L2 at once.
__device__ __forceinline__ int unit_rot(int u, int n, int n_clusters) {
  return n > 0 ? static_cast<int>((static_cast<long long>(u % n_clusters) * n) / n_clusters) : 0;
}
__device__ __forceinline__ int rot_tile(int t0, int n, int i, int rot) {
  int j = i + rot;
  if (j >= n) j -= n;
  return t0 + j;
}

// DW row-split partials, in the layout the drain writes: float4 index of
// [split s][vocab block blk][32-column chunk ch][lane quarter q][float4 v of
// the chunk][lane]: rows blk*128 + 32q + lane, columns 32ch + 4v .. +3.
// Each of a drain warp's stores then covers 512 contiguous bytes.
__host__ __device__ __forceinline__ long long dw_part_index(int s, int blk, int ch, int q, int v, int lane,
                                                           int n_blocks, int nch) {
  return ((((static_cast<long long>(s) * n_blocks + blk) * nch + ch) * 4 + q) * 8 + v) * 32 + lane;
}

// Split-major order: clusters running at the same time share a row range
// of the streamed operand, which then stays in L2.
__device__ __forceinline__ void unit_range(const Params& p, int u, int& blk, int& t0, int& t1) {
  blk = u % p.n_blocks;
  const int s = u / p.n_blocks;
  t0 = static_cast<int>(static_cast<long long>(s) * p.n_tiles / p.split);
  t1 = static_cast<int>(static_cast<long long>(s + 1) * p.n_tiles / p.split);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
               const __grid_constant__ CUtensorMap tm_ys, const Params p) {
  // tm_x: X blocks and tm_y: Y tiles, box 64 x 128 x 4 (four chunks, 64 KB);
  // tm_ys: Y slabs, box 64 x 64 x KC.
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // Z CTA barriers
  uint64_t* zy_full = bars + C::B_ZY_FULL;      // [YSTAGES]
  uint64_t* zy_empty = bars + C::B_ZY_EMPTY;    // [YSTAGES]
  uint64_t* x_free = bars + C::B_X_FREE;        // Z: the previous unit's MMAs no longer read X in TMEM
  uint64_t* x_ready = bars + C::B_X_READY;      // Z: X's tcgen05.cp have completed
  uint64_t* acc_full = bars + C::B_ACC_FULL;    // [2]  Z: z tiles; A: [0] = accumulator done
  uint64_t* acc_empty = bars + C::B_ACC_EMPTY;  // [2]  Z: z tiles; A: [0] = accumulator drained
  uint64_t* p_empty = bars + C::B_P_EMPTY;      // [NPS]  in Z, arrived by A's MMA commit
  // A CTA barriers
  uint64_t* p_full = bars + C::B_P_FULL;        // [NPS]  in A: A's expect_tx + the bytes of Z's st.async
  uint64_t* ay_full = bars + C::B_AY_FULL;      // [ASLOTS] slab slots of the Y ring
  uint64_t* ay_empty = bars + C::B_AY_EMPTY;    // [ASLOTS]
  uint64_t* mma_done = bars + C::B_MMA_DONE;
  uint64_t* rd_full = bars + C::B_RD_FULL;      // FD, in A: the Z epilogue's row records are written
  uint64_t* rd_empty = bars + C::B_RD_EMPTY;    // FD, in Z: the A drain has read them
  uint64_t* stg_full = bars + C::B_STG_FULL;    // [NSTG][2] in Z: the epilogue warps wrote a staging chunk
  uint64_t* stg_empty = bars + C::B_STG_EMPTY;  // [NSTG] in Z: the A CTA has the staged tile (staging free)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 504);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 508);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const bool is_z = (rank == 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::YSTAGES; ++i) {
      mbar_init(zy_full + i, 1);
      mbar_init(zy_empty + i, 1);
    }
    mbar_init(x_free, 1);
    mbar_init(x_ready, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, EPI_WARPS);
    }
    for (int i = 0; i < C::NPS; ++i) {
      mbar_init(p_empty + i, 1);
      mbar_init(p_full + i, 1);
    }
    for (int i = 0; i < C::ASLOTS; ++i) {
      mbar_init(ay_full + i, 1);
      mbar_init(ay_empty + i, 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(rd_full, EPI_WARPS * 32);   // every Z epilogue thread
    for (int i = 0; i < 2 * C::NSTG; ++i) mbar_init(stg_full + i, EPI_WARPS / 2);  // the chunk's 8 warps
    for (int i = 0; i < C::NSTG; ++i) mbar_init(stg_empty + i, 1);                 // the A CTA's acknowledgement
    mbar_init(rd_empty, EPI_WARPS * 32);  // every A drain thread
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  const uint32_t tmem_cols = is_z ? Z_TMEM_COLS : A_TMEM_COLS;
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  // Both CTAs' barriers are initialised before any remote arrive.
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (is_z) {
    // =========================== Z CTA ===========================
    if (warp == TMA_WARP) {
      if (lane == 0) {
        // Ring order: per unit the X block's stages, then per tile the Y
        // tile's stages (chunks past d / 64 read zeros).
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        uint32_t pend = 0, pend_ph[C::YSTAGES] = {};
        const int nst = (p.KC + ZSC - 1) / ZSC;
        auto put = [&](const CUtensorMap* m, int row0, int s4) -> bool {
          if (!mbar_wait(zy_empty + stage, phase ^ 1u, abort_flag, p.status)) return false;
          mbar_expect_tx(zy_full + stage, ZSTAGE);
          tma_load_3d(smem + C::Z_Y + stage * ZSTAGE, m, zy_full + stage, 0, row0, ZSC * s4);
          pend |= 1u << stage;
          pend_ph[stage] = phase;
          if (++stage == C::YSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
          return true;
        };
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
          for (int s4 = 0; s4 < nst && ok; ++s4) ok = put(&tm_x, blk * BM, s4);
          for (int i = 0; i < nt_u && ok; ++i) {
            const int t = bwdk::rot_tile(t0, nt_u, i, rot);
            for (int s4 = 0; s4 < nst && ok; ++s4) ok = put(&tm_y, t * BT, s4);
          }
        }
        if (!ok) {
          const long long c0 = clock64();
          for (int s = 0; s < C::YSTAGES; ++s)
            if (pend & (1u << s))
              while (!mbar_try_wait(smem_u32(zy_full + s), pend_ph[s]) && clock64() - c0 < kWaitLimitCycles) {
              }
        }
      }
    } else if (warp == MMA_WARP) {
      if (lane == 0) {
        int stage = 0, acc = 0;
        uint32_t phase = 0, aph = 0, fph = 0, rph = 0;
        bool ok = true, first = true;
        const int nst = (p.KC + ZSC - 1) / ZSC;
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
          if (!first) {
            // X in TMEM is overwritten only after the previous unit's MMAs.
            umma_commit(x_free);
            ok = mbar_wait(x_free, fph, abort_flag, p.status);
            fph ^= 1u;
            if (!ok) break;
          }
          first = false;
          for (int s4 = 0; s4 < nst && ok; ++s4) {
            ok = mbar_wait(zy_full + stage, phase, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            for (int c = 0; c < ZSC; ++c) {
              const int kc = ZSC * s4 + c;
              if (kc >= p.KC) break;
              const uint32_t xa = smem_u32(smem + C::Z_Y + stage * ZSTAGE + c * CHUNK);
#pragma unroll
              for (int k = 0; k < KB / 16; ++k)
                tmem_cp_128x256b(tmem_base + Z_TMEM_X + static_cast<uint32_t>(kc * 32 + k * 8),
                                 sdesc_sw128(xa + k * 32, 16, 1024));
            }
            umma_commit(zy_empty + stage);
            if (++stage == C::YSTAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(x_ready);
          ok = mbar_wait(x_ready, rph, abort_flag, p.status);
          rph ^= 1u;
          if (!ok) break;
          tc_fence_after();
          for (int i = 0; i < nt_u && ok; ++i) {
            const int t = bwdk::rot_tile(t0, nt_u, i, rot);
            ok = mbar_wait(acc_empty + acc, aph ^ 1u, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BT);
            for (int s4 = 0; s4 < nst && ok; ++s4) {
              ok = mbar_wait(zy_full + stage, phase, abort_flag, p.status);
              if (!ok) break;
              tc_fence_after();
              // The issue loop stays short (descriptors advanced by constant
              // offsets, unrolled): one M=128 N=128 MMA is 64 tensor cycles.
              const uint64_t b0 = sdesc_sw128(smem_u32(smem + C::Z_Y + stage * ZSTAGE), 16, 1024);
              const uint32_t a0 = tmem_base + Z_TMEM_X + static_cast<uint32_t>(s4 * ZSC * 32);
              if (ZSC * (s4 + 1) <= p.KC) {
#pragma unroll
                for (int c = 0; c < ZSC; ++c)
#pragma unroll
                  for (int k = 0; k < KB / 16; ++k)
                    umma_bf16_ts(d_tmem, a0 + static_cast<uint32_t>(c * 32 + k * 8),
                                 b0 + static_cast<uint64_t>((c * CHUNK + k * 32) >> 4), IDESC_Z,
                                 (s4 | c | k) != 0 ? 1u : 0u);
              } else {
                for (int c = 0; c < p.KC - ZSC * s4; ++c)
#pragma unroll
                  for (int k = 0; k < KB / 16; ++k)
                    umma_bf16_ts(d_tmem, a0 + static_cast<uint32_t>(c * 32 + k * 8),
                                 b0 + static_cast<uint64_t>((c * CHUNK + k * 32) >> 4), IDESC_Z,
                                 (s4 | c | k) != 0 ? 1u : 0u);
              }
              umma_commit(zy_empty + stage);
              if (++stage == C::YSTAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit(acc_full + acc);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
          }
        }
        umma_commit(mma_done);
        const long long c0 = clock64();
        while (!mbar_try_wait(smem_u32(mma_done), 0) && clock64() - c0 < kWaitLimitCycles) {
        }
      }
    } else if (warp == FWD_WARP) {
      if (lane == 0) {
        // ---- P forwarder: staging copy -> the A CTA's P slot ----
        // Per tile, each 16 KB column chunk goes in one bulk DSMEM copy that
        // completes the slot's mbarrier in the A CTA (which expects the whole
        // tile), once that slot's previous tile has been consumed.  The A
        // CTA acknowledges each landed tile on stg_empty, which frees the
        // staging copy for the epilogue.
        const uint32_t peer_p = mapa_shared(smem_u32(smem + C::A_P), 1);
        const uint32_t peer_pfull = mapa_shared(smem_u32(p_full), 1);
        const uint32_t stg = smem_u32(smem + C::Z_STG);
        int slot = 0;
        uint32_t sph = 0;
        int issued = 0;  // tiles sent; tile n uses staging copy n % NSTG
        bool ok = true;
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          for (int i = 0; i < t1 - t0 && ok; ++i) {
            const int set = issued % C::NSTG;
            const uint32_t use_ph = static_cast<uint32_t>(issued / C::NSTG) & 1u;
            for (int h = 0; h < 2 && ok; ++h) {
              ok = mbar_wait(stg_full + 2 * set + h, use_ph, abort_flag, p.status);
              if (ok && h == 0) ok = mbar_wait<true>(p_empty + slot, sph ^ 1u, abort_flag, p.status);
              if (ok)
                bulk_copy_to_peer(peer_p + static_cast<uint32_t>(slot) * P_SLOT + static_cast<uint32_t>(h) * CHUNK,
                                  stg + static_cast<uint32_t>(2 * set + h) * CHUNK, CHUNK,
                                  peer_pfull + static_cast<uint32_t>(slot) * 8u);
            }
            if (!ok) break;
            ++issued;
            if (++slot == C::NPS) {
              slot = 0;
              sph ^= 1u;
            }
          }
        }
        if (ok) {
          // Every staging copy's last acknowledgement: no copy is in flight after them.
          for (int set = 0; set < C::NSTG && set < issued && ok; ++set) {
            const int uses = (issued - set + C::NSTG - 1) / C::NSTG;
            ok = mbar_wait<true>(stg_empty + set, static_cast<uint32_t>(uses - 1) & 1u, abort_flag, p.status);
          }
        } else {
          // Let copies already issued land before this CTA can leave.
          const long long c0 = clock64();
          while (clock64() - c0 < 200000) {
          }
        }
      }
    } else {
      // ---- Z epilogue: z tile -> P tile in a staging copy ----
      // Warp w reads TMEM lanes 32 (w % 4) .. +31 (its 32 rows) and columns
      // 32 (w / 4) .. +31 of each tile: one 32-column chunk per warp and tile,
      // four warps per scheduler so that TMEM loads, math and the stores of
      // different warps overlap.
      const int q = warp & 3;
      const int cq = warp >> 2;     // 32-column group of the tile
      const int m = q * 32 + lane;  // row of the P tile (= TMEM lane)
      EpiConst kc;
      kc.m1 = make_float2(-1.0f, -1.0f);
      kc.cl2e2 = make_float2(p.cl2e, p.cl2e);
      kc.invc2 = make_float2(p.inv_c, p.inv_c);
      kc.xlim = p.xlim;
      kc.inv_c = p.inv_c;
      kc.cl2e = p.cl2e;
      const float kNegInf = __int_as_float(0xff800000);
      // DW: row data of the warp's 32 columns (lane j holds column j):
      // -lse log2(e) (-inf for rows that do not count), the block lane of the
      // row's target, and its p_t - 1.  pf_* is the next tile's, fetched early.
      float cur_nl = kNegInf, pf_nl = kNegInf;
      int cur_hit = -1, pf_hit = -1;
      float cur_pm1 = 0.f, pf_pm1 = 0.f;
      const int use_pm1 = p.nll_in != nullptr;
      const uint32_t stg = smem_u32(smem + C::Z_STG);
      const uint32_t peer_rd_full = mapa_shared(smem_u32(rd_full), 1);
      int acc = 0;
      uint32_t aph = 0;
      int staged = 0;  // tiles staged; tile n uses staging copy n % NSTG
      bool ok = true;
      int fd_units = 0;
      for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
        int blk, t0, t1;
        unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
        // DH: this thread's row data.
        float nl_row = kNegInf;
        long long trow = -1;
        float pm1_row = 0.f;
        if (MODE == DH) {
          const int row = blk * BM + m;
          if (row < p.N && (!p.mask || p.mask[row])) {
            const long long tt = p.tgt[row];
            nl_row = -p.lse[row] * kLog2e;
            if (use_pm1) pm1_row = expm1f(-p.nll_in[row]);
            if (tt >= 0 && tt < p.V) trow = tt;
            else if (cq == 0) atomicOr(p.status, ST_EDATA);
          }
        }
        // FD: this thread's row data and its running sums over the unit.
        int fd_flags = 0;
        // The row's sum of e^s over its non-target columns, compensated in
        // fp32 (Neumaier: s_hi + s_lo carries about twice fp32's precision);
        // B300's fp64 pipe is too narrow for an add per chunk and thread.
        float s_hi = 0.f, s_lo = 0.f;
        FdTarget rec_tg{0.f, 0.f};
        if (MODE == FD) {
          const int row = blk * BM + m;
          if (row < p.N && (!p.mask || p.mask[row])) {
            const long long tt = p.tgt[row];
            nl_row = 0.f;
            fd_flags = FL_LIVE;
            if (tt >= 0 && tt < p.V) {
              trow = tt;
              fd_flags |= FL_TVALID;
            } else if (cq == 0) {
              atomicOr(p.status, ST_EDATA);
            }
          }
        }
        const long long vbase = static_cast<long long>(blk) * BM;
        // DW: row data of tile t is fetched into registers one tile ahead.
        auto fetch_dw = [&](int t) {
          const int row = t * BT + cq * 32 + lane;
          float nl = kNegInf;
          int hl = -1;
          float q1 = 0.f;
          if (row < p.N) {
            const uint8_t mk = p.mask ? p.mask[row] : uint8_t(1);
            const long long tt = p.tgt[row];
            const float l = p.lse[row];
            if (mk) {
              nl = -l * kLog2e;
              if (tt < 0 || tt >= p.V) atomicOr(p.status, ST_EDATA);
              else if (tt >= vbase && tt < vbase + BM) hl = static_cast<int>(tt - vbase);
              if (hl >= 0 && use_pm1) q1 = expm1f(-p.nll_in[row]);
            }
          }
          pf_nl = nl;
          pf_hit = hl;
          pf_pm1 = q1;
        };
        if (MODE == DW && nt_u > 0) fetch_dw(bwdk::rot_tile(t0, nt_u, 0, rot));
        for (int i = 0; i < nt_u; ++i) {
            const int t = bwdk::rot_tile(t0, nt_u, i, rot);
          bool hit_any = false;
          if (MODE == DW) {
            cur_nl = pf_nl;
            cur_hit = pf_hit;
            cur_pm1 = pf_pm1;
            hit_any = __any_sync(0xffffffffu, pf_hit >= 0);
            if (i + 1 < nt_u) fetch_dw(bwdk::rot_tile(t0, nt_u, i + 1, rot));
          }
          ok = mbar_wait(acc_full + acc, aph, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          uint32_t r[32];
          tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BT + cq * 32), r);
          tmem_ld_wait();
          reg_fence32(r);
          // The chunk is in registers: release the accumulator buffer.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + acc);
          acc ^= 1;
          if (acc == 0) aph ^= 1u;
          // Gradient (or FD tile) of the chunk, packed to bf16.
          uint32_t packed[16];
          const int cbase = t * BT + cq * 32;  // first column of the chunk (vocab index in DH, FD)
          if (MODE == DH) {
            const int lim = min(32, p.V - cbase);
            const long long relw = trow - cbase;
            const int rel = (relw >= 0 && relw < 32) ? static_cast<int>(relw) : -1;
            if (__any_sync(0xffffffffu, rel >= 0))
              g_chunk_dh<true>(r, kc, -nl_row, rel, lim, use_pm1, pm1_row, packed);
            else
              g_chunk_dh<false>(r, kc, -nl_row, -1, lim, use_pm1, pm1_row, packed);
          } else if (MODE == FD) {
            const int lim = min(32, p.V - cbase);
            const long long relw = trow - cbase;
            const int rel = (relw >= 0 && relw < 32) ? static_cast<int>(relw) : -1;
            FdTarget tg{0.f, 0.f};
            float cs;
            if (__any_sync(0xffffffffu, rel >= 0))
              cs = g_chunk_fd<true>(r, kc, nl_row, rel, lim, packed, tg);
            else
              cs = g_chunk_fd<false>(r, kc, nl_row, -1, lim, packed, tg);
            const float sn = s_hi + cs;
            s_lo += (fabsf(s_hi) >= fabsf(cs)) ? ((s_hi - sn) + cs) : ((cs - sn) + s_hi);
            s_hi = sn;
            if (rel >= 0) {
              rec_tg = tg;
              fd_flags |= FL_HIT;
            }
          } else {
            if (hit_any)
              g_chunk_dw<true>(r, kc, cur_nl, cur_hit, m, use_pm1, cur_pm1, packed);
            else
              g_chunk_dw<false>(r, kc, cur_nl, cur_hit, m, use_pm1, cur_pm1, packed);
          }
          // Four swizzled 16-byte stores into the staging copy (the P slot
          // layout), once that copy's previous tile has reached the A CTA;
          // the forwarder warp then sends each 64-column chunk in one bulk
          // copy.
          const int set = staged % C::NSTG;
          ok = mbar_wait<true>(stg_empty + set, (static_cast<uint32_t>(staged / C::NSTG) & 1u) ^ 1u, abort_flag,
                               p.status);
          if (!ok) break;
          const uint32_t dst_row =
              stg + static_cast<uint32_t>(2 * set + (cq >> 1)) * CHUNK + static_cast<uint32_t>(m) * 128u;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t unit = static_cast<uint32_t>((cq & 1) * 4 + v);
            const uint32_t addr = dst_row + ((unit ^ static_cast<uint32_t>(m & 7)) << 4);
            st_shared_v4(addr, packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
          }
          fence_proxy_async_smem();  // visible to the bulk copy (async proxy)
          __syncwarp();
          if (lane == 0) mbar_arrive(stg_full + 2 * set + (cq >> 1));
          ++staged;
        }
        if (MODE == FD) {
          // Row record for the A drain, once it has read the previous one.
          if (!ok) break;
          if (fd_units > 0) {
            ok = mbar_wait<true>(rd_empty, static_cast<uint32_t>(fd_units - 1) & 1u, abort_flag, p.status);
            if (!ok) break;
          }
          // Global stores, ordered before the cluster-scope release arrival.
          uint4* rec = p.fd_rec + (static_cast<size_t>(cluster * NREC_GROUPS + cq) * BM + m) * 2;
          rec[0] = make_uint4(__float_as_uint(s_hi + s_lo), 0u, __float_as_uint(rec_tg.e), __float_as_uint(rec_tg.om));
          rec[1] = make_uint4(static_cast<uint32_t>(trow), static_cast<uint32_t>(fd_flags), 0u, 0u);
          mbar_arrive_cluster(peer_rd_full);
          ++fd_units;
        }
      }
    }
  } else {
    // =========================== A CTA ===========================
    if (warp == TMA_WARP) {
      if (lane == 0) {
        // The Y tiles arrive in slabs of 64 rows x d (one load each) through
        // a ring of ASLOTS slab slots.
        int rs = 0;
        uint32_t rph = 0;
        bool ok = true;
        uint32_t pend = 0, pend_ph[C::ASLOTS] = {};
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
          for (int i = 0; i < nt_u && ok; ++i) {
            const int t = bwdk::rot_tile(t0, nt_u, i, rot);
            for (int sl = 0; sl < NSLAB; ++sl) {
              ok = mbar_wait(ay_empty + rs, rph ^ 1u, abort_flag, p.status);
              if (!ok) break;
              mbar_expect_tx(ay_full + rs, p.KC * SLAB_CHUNK);
              tma_load_3d(smem + C::A_Y + rs * p.KC * SLAB_CHUNK, &tm_ys, ay_full + rs, 0, t * BT + sl * SLAB_ROWS, 0);
              pend |= 1u << rs;
              pend_ph[rs] = rph;
              if (++rs == C::ASLOTS) {
                rs = 0;
                rph ^= 1u;
              }
            }
          }
        }
        if (!ok) {
          const long long c0 = clock64();
          for (int s = 0; s < C::ASLOTS; ++s)
            if (pend & (1u << s))
              while (!mbar_try_wait(smem_u32(ay_full + s), pend_ph[s]) && clock64() - c0 < kWaitLimitCycles) {
              }
        }
      }
    } else if (warp == MMA_WARP) {
      if (lane == 0) {
        uint32_t rph = 0, sph = 0, dph = 0;
        int slot = 0, rs = 0;
        bool ok = true;
        // The accumulator's d columns in two N halves of nh0 and nh1 chunks.
        const int nh0 = (p.KC + 1) / 2;
        const int nh1 = p.KC - nh0;
        const uint32_t idesc_h0 = idesc_bf16_f32(128, 64 * nh0, false, true);
        const uint32_t idesc_h1 = idesc_bf16_f32(128, 64 * (nh1 > 0 ? nh1 : 1), false, true);
        // Each P slot completes when all its bytes (st.async from the Z CTA)
        // have landed: arm every slot for its first use.
        for (int i = 0; i < C::NPS; ++i) mbar_expect_tx(p_full + i, P_SLOT);
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
          ok = mbar_wait(acc_empty, dph ^ 1u, abort_flag, p.status);  // accumulator drained
          dph ^= 1u;
          if (!ok) break;
          tc_fence_after();
          for (int i = 0; i < nt_u && ok; ++i) {
            const int t = bwdk::rot_tile(t0, nt_u, i, rot);
            ok = mbar_wait<true>(p_full + slot, sph, abort_flag, p.status);
            if (!ok) break;
            mbar_expect_tx(p_full + slot, P_SLOT);  // arm the slot's next use
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t pdesc = sdesc_sw128(smem_u32(smem + C::A_P + slot * P_SLOT), 16, 1024);
            for (int sl = 0; sl < NSLAB && ok; ++sl) {
              ok = mbar_wait(ay_full + rs, rph, abort_flag, p.status);
              if (!ok) break;
              tc_fence_after();
              // The slab's four K steps of 16 rows (2 KB apart); P: the chunk
              // of K columns 64 sl .. +63, 16 kk + .. (32 bytes per step).
              // MN-major B: N = 64 nh columns of d in chunks 8 KB apart inside
              // the slab.
              const uint64_t bd0 = sdesc_sw128(smem_u32(smem + C::A_Y + rs * p.KC * SLAB_CHUNK), SLAB_CHUNK, 1024);
              const int pc0 = sl * SLAB_ROWS;  // first P column (K row) of the slab
              const uint64_t ad0 = pdesc + static_cast<uint64_t>(((pc0 / KB) * CHUNK + (pc0 % KB) * 2) >> 4);
#pragma unroll
              for (int kk = 0; kk < SLAB_ROWS / 16; ++kk) {
                const uint32_t accf = (i != 0 || sl != 0 || kk != 0) ? 1u : 0u;
                const uint64_t ad = ad0 + static_cast<uint64_t>((kk * 32) >> 4);
                const uint64_t bd = bd0 + static_cast<uint64_t>((kk * 2048) >> 4);
                umma_bf16(tmem_base, ad, bd, idesc_h0, accf);
                if (nh1 > 0)
                  umma_bf16(tmem_base + static_cast<uint32_t>(64 * nh0), ad,
                            bd + static_cast<uint64_t>((nh0 * SLAB_CHUNK) >> 4), idesc_h1, accf);
              }
              umma_commit(ay_empty + rs);
              if (++rs == C::ASLOTS) {
                rs = 0;
                rph ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit_mc(p_empty + slot, static_cast<uint16_t>(1u << 0));  // P slot free (Z CTA)
            if (++slot == C::NPS) {
              slot = 0;
              sph ^= 1u;
            }
          }
          if (ok) umma_commit(acc_full);  // accumulator of this unit complete
        }
        umma_commit(mma_done);
        const long long c0 = clock64();
        while (!mbar_try_wait(smem_u32(mma_done), 0) && clock64() - c0 < kWaitLimitCycles) {
        }
      }
    } else if (warp == FWD_WARP) {
      if (lane == 0) {
        // ---- P acknowledgements: each tile's bytes have landed ----
        // The Z CTA's staging copy is free once the bulk copies into the P
        // slot have completed; the slots are visited in the MMA warp's order.
        const uint32_t z_stg_empty = mapa_shared(smem_u32(stg_empty), 0);
        int slot = 0, n = 0;
        uint32_t sph = 0;
        bool ok = true;
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          for (int i = 0; i < t1 - t0 && ok; ++i) {
            ok = mbar_wait<true>(p_full + slot, sph, abort_flag, p.status);
            if (!ok) break;
            mbar_arrive_cluster(z_stg_empty + static_cast<uint32_t>(n % C::NSTG) * 8u);
            ++n;
            if (++slot == C::NPS) {
              slot = 0;
              sph ^= 1u;
            }
          }
        }
      }
    } else {
      // ---- A drain: accumulator -> dh / dW ----
      // Warp w drains TMEM lanes 32 (w % 4) .. +31 and the 32-column chunks
      // w / 4, w / 4 + 4, ... of the d columns.
      const int q = warp & 3;
      const int part = warp >> 2;
      const int m = q * 32 + lane;
      constexpr int NPART = EPI_WARPS / 4;
      uint32_t fph = 0, rph = 0;
      const uint32_t z_rd_empty = mapa_shared(smem_u32(rd_empty), 0);
      for (int u = cluster; u < p.n_units; u += n_clusters) {
        int blk, t0, t1;
        unit_range(p, u, blk, t0, t1);
          const int nt_u = t1 - t0, rot = bwdk::unit_rot(u, nt_u, n_clusters);
        const int row = blk * BM + m;  // DH, FD: token row; DW: vocab row
        const int nch = p.d / 32;      // 32-column chunks of the accumulator
        // FD: the row's scale alpha, target term beta W_t, and the forward's
        // outputs, from the Z epilogue's records of the row (one per column
        // group, in group order).
        float alpha = 0.f, beta = 0.f;
        long long trow = -1;
        if (MODE == FD) {
          if (!mbar_wait<true>(rd_full, rph, abort_flag, p.status)) break;
          rph ^= 1u;
          // The row's sum of e^s over its non-target columns (the column
          // groups' sums added in group order), the target's e^{s_t} and
          // 1 - tanh_t^2; the scales and the logarithms in fp32 (a few ulp,
          // and none of B300's slow fp64 arithmetic in front of the drain).
          float S_other = 0.f;
          int flags = 0;
          uint32_t tsel = 0;
          float et = 0.f, om = 0.f;
#pragma unroll
          for (int g = 0; g < NREC_GROUPS; ++g) {
            // After the cluster-scope acquire of rd_full; read at L2.
            const uint4* ra = p.fd_rec + (static_cast<size_t>(cluster * NREC_GROUPS + g) * BM + m) * 2;
            const uint4 a0 = __ldcg(ra), a1 = __ldcg(ra + 1);
            S_other += __uint_as_float(a0.x);
            flags |= static_cast<int>(a1.y);
            tsel = a1.x;
            if (a1.y & FL_HIT) {
              et = __uint_as_float(a0.z);
              om = __uint_as_float(a0.w);
            }
          }
          mbar_arrive_cluster(z_rd_empty);
          const bool tv = (flags & FL_TVALID) != 0;
          const float S = tv ? S_other + et : S_other;
          if (flags & FL_LIVE) {
            alpha = -p.w / S;
            if (tv) {
              // w (p_t - 1)(1 - tanh_t^2), p_t - 1 = -S_other / S (no cancellation).
              beta = -p.w * (S_other / S) * om;
              trow = static_cast<long long>(static_cast<int>(tsel));
            }
          }
          if (part == 0 && row < p.N) {
            float nll = 0.f, lse = 0.f;
            if (flags & FL_LIVE) {
              lse = logf(S);
              nll = tv ? nll_from_sums(S_other, et) : __int_as_float(0x7fc00000);
            }
            p.nll[row] = nll;
            if (p.lse_out) p.lse_out[row] = lse;
          }
        }
        // FD: W_t's columns of chunk ch (bf16), fetched one chunk ahead.
        uint4 wcur[4], wnxt[4];
        auto load_w = [&](int ch, uint4(&dst)[4]) {
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
          if (trow >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(p.W + trow * p.d + ch * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = __ldg(src + v);
          }
        };
        if (MODE == FD && part < nch) load_w(part, wcur);
        if (!mbar_wait(acc_full, fph, abort_flag, p.status)) break;
        fph ^= 1u;
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
        for (int ch = part; ch < nch; ch += NPART) {
          if (MODE == FD && ch + NPART < nch) load_w(ch + NPART, wnxt);
          uint32_t r[32];
          tmem_ld32(tb + ch * 32, r);
          tmem_ld_wait();
          reg_fence32(r);
          const int col = ch * 32;
          if (MODE == FD) {
            if (row < p.N) {
              const uint32_t* wb = reinterpret_cast<const uint32_t*>(wcur);
              __align__(16) __nv_bfloat16 o[32];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float wl = __uint_as_float(wb[j] << 16);
                const float wh = __uint_as_float(wb[j] & 0xffff0000u);
                o[2 * j] = __float2bfloat16_rn(fmaf(alpha, __uint_as_float(r[2 * j]), beta * wl));
                o[2 * j + 1] = __float2bfloat16_rn(fmaf(alpha, __uint_as_float(r[2 * j + 1]), beta * wh));
              }
              uint4* dst = reinterpret_cast<uint4*>(p.dh + static_cast<long long>(row) * p.ldh + col);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = reinterpret_cast<const uint4*>(o)[v];
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) wcur[v] = wnxt[v];
          } else if (MODE == DH) {
            if (row < p.N) {
              __align__(16) __nv_bfloat16 o[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float2bfloat16_rn(p.w * __uint_as_float(r[j]));
              uint4* dst = reinterpret_cast<uint4*>(p.dh + static_cast<long long>(row) * p.ldh + col);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = reinterpret_cast<const uint4*>(o)[v];
            }
          } else {
            if (row < p.V) {
              if (p.split == 1) {
                float4* dst = reinterpret_cast<float4*>(p.dW + static_cast<long long>(row) * p.d + col);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  float4 a = make_float4(p.w * __uint_as_float(r[4 * v]), p.w * __uint_as_float(r[4 * v + 1]),
                                         p.w * __uint_as_float(r[4 * v + 2]), p.w * __uint_as_float(r[4 * v + 3]));
                  if (p.accumulate) {
                    const float4 b = dst[v];
                    a.x += b.x;
                    a.y += b.y;
                    a.z += b.z;
                    a.w += b.w;
                  }
                  dst[v] = a;
                }
              } else {
                // The partial in the drain's own layout (dw_part_index): each
                // store instruction writes 512 contiguous bytes.
                const int s = u / p.n_blocks;
                float4* dst = reinterpret_cast<float4*>(p.dw_part) + dw_part_index(s, blk, ch, q, 0, lane, p.n_blocks, nch);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v * 32] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                            __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // No CTA leaves while its peer may still touch its shared memory.
  cluster_arrive();
  cluster_wait();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// dW = (accumulate ? dW : 0) + w * sum_{s < split} part[s], in split order,
// from the drain's partial layout (dw_part_index).  One block per (vocab
// block, 32-column chunk): its 256 threads add the splits' float4 planes
// (reads coalesced across the lanes) into a shared-memory tile, then write
// the chunk's 128 rows x 128 bytes of dW (8 threads per row: coalesced).
__global__ void __launch_bounds__(256) dw_split_reduce_kernel(const float4* __restrict__ part, int split, int n_blocks,
                                                              int nch, int V, int d, float w, int accumulate,
                                                              float* __restrict__ dW) {
  __shared__ float4 tile[4 * 8][33];  // [q * 8 + v][lane], padded against bank conflicts
  const int blk = blockIdx.x / nch;
  const int ch = blockIdx.x - blk * nch;
  const long long sstride = static_cast<long long>(n_blocks) * nch * 4 * 256;
  const float4* src = part + dw_part_index(0, blk, ch, 0, 0, 0, n_blocks, nch);
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int e = it * 256 + threadIdx.x;  // (q, v, lane) of the chunk's 1024 float4
    float4 b[MAX_SPLIT];
#pragma unroll
    for (int k = 0; k < MAX_SPLIT; ++k)
      if (k < split) b[k] = src[k * sstride + e];
    float4 s = b[0];
#pragma unroll
    for (int k = 1; k < MAX_SPLIT; ++k) {
      if (k < split) {
        s.x += b[k].x;
        s.y += b[k].y;
        s.z += b[k].z;
        s.w += b[k].w;
      }
    }
    tile[e >> 5][e & 31] = make_float4(w * s.x, w * s.y, w * s.z, w * s.w);
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int e = it * 256 + threadIdx.x;
    const int r = e >> 3, v = e & 7;  // row of the block, float4 of the chunk
    const int row = blk * BM + r;
    if (row >= V) continue;
    float4 o = tile[(r >> 5) * 8 + v][r & 31];
    float4* dst = reinterpret_cast<float4*>(dW + static_cast<long long>(row) * d + ch * 32) + v;
    if (accumulate) {
      const float4 a = *dst;
      o.x += a.x;
      o.y += a.y;
      o.z += a.z;
      o.w += a.w;
    }
    *dst = o;
  }
}

inline long long cdivll(long long a, long long b) { return (a + b - 1) / b; }

// Row splits for the vocab-stationary (dW) pass: enough units to fill the
// clusters evenly, at most MAX_SPLIT (each split writes a [V, d] partial).
inline int choose_split(long long N, long long V, int clusters) {
  const long long nb = cdivll(V, BM);
  const long long nt = cdivll(N, BT);
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= MAX_SPLIT && s <= nt; ++s) {
    const long long units = nb * s;
    const double waves = static_cast<double>(cdivll(units, clusters));
    const double cost = waves / s * (1.0 + 0.01 * (s - 1));  // small penalty for the partial traffic
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// FD row-record area for N rows: one 16 KB area per cluster of the launch.
inline size_t fd_rec_bytes(long long N) {
  const long long blocks = cdivll(N, BM);
  return static_cast<size_t>(blocks < kFdRecClusters ? blocks : kFdRecClusters) * kFdRecClusterBytes;
}

inline size_t scratch_bytes(long long N, long long V, long long d) {
  const long long nt = cdivll(N, BT);
  const long long s = nt < MAX_SPLIT ? nt : MAX_SPLIT;
  if (s <= 1) return 0;
  return static_cast<size_t>(s) * static_cast<size_t>(cdivll(V, BM) * BM) * static_cast<size_t>(d) * 4u;
}

inline int setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<DH>::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_kernel<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<DW>::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_kernel<FD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<FD>::SMEM_BYTES);
  if (e != cudaSuccess) {
    set_last_error(std::string("cudaFuncSetAttribute(bwd): ") + cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

// Co-resident 2-CTA clusters for this kernel on device `dev` (cached per
// device), for the mode with the most shared memory (every mode runs one CTA
// per SM).
inline int max_clusters(int dev, int sms) {
  static int cached[64] = {};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<FD>::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, bwd_kernel<FD>, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = sms / 2;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

template <int MODE>
inline int launch_mode(const CUtensorMap& tx, const CUtensorMap& ty, const CUtensorMap& tys, const Params& p,
                       int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Cfg<MODE>::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_kernel<MODE>, tx, ty, tys, p);
  if (e != cudaSuccess) {
    set_last_error(std::string("bwd_kernel launch: ") + cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

inline int launch(const uint16_t* h, long long ldh, const uint16_t* W, long long N, long long V, long long d,
                  const int64_t* tgt, const uint8_t* mask, float c, const float* lse, const float* nll, float w,
                  uint16_t* dh, float* dW, int accumulate, unsigned* status, void* scratch, int dev, int sms,
                  cudaStream_t s) {
  const uint32_t kc = static_cast<uint32_t>(d / KB);
  CUtensorMap tm_hx, tm_wx, tm_hy, tm_wy, tm_hs, tm_ws;
  if (int rc = make_map_bf16_3d(&tm_hx, h, d, N, ldh * 2, BM, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_wx, W, d, V, d * 2, BM, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_hy, h, d, N, ldh * 2, BT, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_wy, W, d, V, d * 2, BT, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_hs, h, d, N, ldh * 2, SLAB_ROWS, kc); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_ws, W, d, V, d * 2, SLAB_ROWS, kc); rc) return rc;
  const int clusters_max = max_clusters(dev, sms);
  Params p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.d = static_cast<int>(d);
  p.KC = static_cast<int>(d / KB);
  p.tgt = tgt;
  p.mask = mask;
  p.lse = lse;
  p.nll_in = nll;
  p.w = -w;  // the P tiles hold -G
  if (c > 0.0f) {
    p.inv_c = 1.0f / c;
    p.cl2e = c * kLog2e;
    p.xlim = kTanhXmax;
  } else {
    // No cap (softcap 0): the epilogue runs with c = 1e30, where in fp32
    // tanh(z/c) = z/c to within the SFU's relative error, so that
    // c log2(e) tanh(z/c) = z log2(e) to that error and one rounding of the
    // two constants, tanh^2 underflows so 1 - tanh^2 = 1, and the range
    // check never sends a chunk to the exact slow path.
    const float ce = 1e30f;
    p.inv_c = 1.0f / ce;
    p.cl2e = ce * kLog2e;
    p.xlim = HUGE_VALF;
  }
  p.status = status;
  if (dh) {
    Params q = p;
    q.n_blocks = static_cast<int>(cdivll(N, BM));
    q.n_tiles = static_cast<int>(cdivll(V, BT));
    q.split = 1;
    q.n_units = q.n_blocks;
    q.dh = reinterpret_cast<__nv_bfloat16*>(dh);
    q.ldh = ldh;
    const int cl = static_cast<int>(q.n_units < clusters_max ? q.n_units : clusters_max);
    if (int rc = launch_mode<DH>(tm_hx, tm_wy, tm_ws, q, cl, s); rc) return rc;
  }
  if (dW) {
    Params q = p;
    q.n_blocks = static_cast<int>(cdivll(V, BM));
    q.n_tiles = static_cast<int>(cdivll(N, BT));
    q.split = choose_split(N, V, clusters_max);
    q.n_units = q.n_blocks * q.split;
    q.dW = dW;
    q.accumulate = accumulate;
    q.V_pad = static_cast<int>(cdivll(V, BM) * BM);
    q.dw_part = static_cast<float*>(scratch);
    const int cl = static_cast<int>(q.n_units < clusters_max ? q.n_units : clusters_max);
    if (int rc = launch_mode<DW>(tm_wx, tm_hy, tm_hs, q, cl, s); rc) return rc;
    if (q.split > 1) {
      const int blocks = q.n_blocks * static_cast<int>(d / 32);
      count_launches(1);
      dw_split_reduce_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(scratch), q.split, q.n_blocks,
                                                    static_cast<int>(d / 32), static_cast<int>(V), static_cast<int>(d),
                                                    p.w, accumulate, dW);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) {
        set_last_error(std::string("dw_split_reduce launch: ") + cudaGetErrorString(e));
        return 3;
      }
    }
  }
  return 0;
}

// Forward + dh in one pass (FD mode): nll and lse (nullable) [N] fp32, dh
// [N, ldh] bf16, for L = grad_scale * sum of nll over the scored rows.
inline int launch_fd(const uint16_t* h, long long ldh, const uint16_t* W, long long N, long long V, long long d,
                     const int64_t* tgt, const uint8_t* mask, float c, float grad_scale, float* nll, float* lse,
                     uint16_t* dh, unsigned* status, void* rec, int dev, int sms, cudaStream_t s) {
  CUtensorMap tm_hx, tm_wy, tm_ws;
  if (int rc = make_map_bf16_3d(&tm_hx, h, d, N, ldh * 2, BM, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_wy, W, d, V, d * 2, BT, ZSC); rc) return rc;
  if (int rc = make_map_bf16_3d(&tm_ws, W, d, V, d * 2, SLAB_ROWS, static_cast<uint32_t>(d / KB)); rc) return rc;
  const int clusters_max = max_clusters(dev, sms);
  Params p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.d = static_cast<int>(d);
  p.KC = static_cast<int>(d / KB);
  p.tgt = tgt;
  p.mask = mask;
  p.inv_c = 1.0f / c;
  p.c = c;
  p.cl2e = c * kLog2e;
  p.w = grad_scale;
  p.xlim = kTanhXmax;
  p.status = status;
  p.W = reinterpret_cast<const __nv_bfloat16*>(W);
  p.nll = nll;
  p.lse_out = lse;
  p.dh = reinterpret_cast<__nv_bfloat16*>(dh);
  p.ldh = ldh;
  p.n_blocks = static_cast<int>(cdivll(N, BM));
  p.n_tiles = static_cast<int>(cdivll(V, BT));
  p.split = 1;
  p.n_units = p.n_blocks;
  p.fd_rec = static_cast<uint4*>(rec);
  int cl = static_cast<int>(p.n_units < clusters_max ? p.n_units : clusters_max);
  if (cl > kFdRecClusters) cl = kFdRecClusters;
  return launch_mode<FD>(tm_hx, tm_wy, tm_ws, p, cl, s);
}

}  // namespace bwdk
}  // namespace lmce
