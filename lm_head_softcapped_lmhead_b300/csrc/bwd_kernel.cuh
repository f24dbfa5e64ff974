// bwd_kernel.cuh -- backward of the fused tied-LM-head + softcapped CE:
//   G_ij = (p_ij - [j == t_i]) (1 - tanh^2(z_ij / c)),  p_ij = e^{s_ij - lse_i}
//   dh = w G W            (rows stationary, "DH" mode)
//   dW (+)= w G^T h       (vocab stationary, "DW" mode)
// Chain rule of nll_i = lse_i - s_{i,t_i} through s = c tanh(z/c), for the
// training step of "parameter-golf: ... Where Model Size Becomes the Game",
// section "The Baseline Is a Map, Not the Destination" (loss.backward()).
//
// A [128 rows x 512] fp32 accumulator fills all of an SM's TMEM, so the logit
// tile and the accumulator cannot share one SM.  Each stationary block is
// therefore handled by a cluster of two CTAs:
//  * rank 0, the Z CTA: keeps the stationary operand X (128 x d bf16) in
//    shared memory, streams the other operand Y in 128-row tiles, computes
//    z = X Y^T (tcgen05, M=128 N=128, double-buffered in TMEM), and turns each
//    z tile into the bf16 tile P = G (DH) or G^T (DW) in the epilogue; P is
//    stored straight into the peer CTA's shared memory (DSMEM), in the
//    128B-swizzled K-major layout the MMA reads.
//  * rank 1, the A CTA: loads the same Y tile (as the MN-major B operand) and
//    accumulates acc (128 x d fp32, all 512 TMEM columns) += P Y with
//    tcgen05 M=128 N=256; after the last tile it scales by w and writes dh
//    (bf16) or dW (fp32, added or stored; or a partial for a later ordered
//    reduction when the rows are split across several clusters).
// The logits and G never leave the two SMs.  Every wait is bounded.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <string>

#include "ptx.cuh"
#include "softcap_math.cuh"

namespace lmce {
int make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
                  uint32_t box_inner, uint32_t box_outer);
void set_last_error(const std::string& s);
void count_launches(unsigned n);

namespace bwdk {

enum Mode : int { DH = 0, DW = 1 };

constexpr int BM = 128;   // stationary block (TMEM lanes)
constexpr int BT = 128;   // streamed tile (z columns; K of the accumulation)
constexpr int KB = 64;    // K elements per chunk
constexpr int MAX_KC = 8; // d <= 512
constexpr int YSTAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr uint32_t CHUNK = 128 * KB * 2;  // 16 KB: 128 rows x 64 bf16
// Z CTA layout
constexpr uint32_t Z_X = 0;
constexpr uint32_t Z_Y = Z_X + MAX_KC * CHUNK;          // ring of YSTAGES chunks
constexpr uint32_t Z_SIDE = Z_Y + YSTAGES * CHUNK;      // DW: per-warp row data (64 lse2 + 64 hit)
constexpr uint32_t Z_END = Z_SIDE + 8 * 64 * 8;
// A CTA layout
constexpr uint32_t A_Y = 0;                             // one full Y tile: MAX_KC chunks
constexpr uint32_t A_P = A_Y + MAX_KC * CHUNK;          // 2 P slots of 128 x 128 bf16
constexpr uint32_t P_SLOT = 2 * CHUNK;                  // 32 KB
constexpr uint32_t A_END = A_P + 2 * P_SLOT;
constexpr uint32_t BAR_OFF = (Z_END > A_END ? Z_END : A_END);
constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;
constexpr uint32_t Z_TMEM_COLS = 256;
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
  float inv_c, cl2e, w;
  __nv_bfloat16* dh;    // DH output [N, ldh]
  long long ldh;
  float* dW;            // DW output [V, d]
  int accumulate;
  float* dw_part;       // DW split partials [split][V_pad][d]
  int V_pad;
  unsigned* status;
};

// Gradient for 32 columns of one lane-row.  DH: column = vocab, per-thread
// lse2 / rel (target column relative to the chunk, or -1).  Writes 16 packed
// bf16x2 words.  Columns >= lim are forced to 0.
template <bool kHit>
__device__ __forceinline__ void g_chunk_dh(const uint32_t (&r)[32], float inv_c, float cl2e, float lse2, int rel,
                                           int lim, uint32_t (&out)[16]) {
  float xmax = 0.f;
  float g[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x = __uint_as_float(r[j]) * inv_c;
    xmax = fmaxf(xmax, fabsf(x));
    const float th = tanh_poly(x);
    const float p = ex2_approx(fmaf(th, cl2e, -lse2));
    const float tau = fmaf(-th, th, 1.0f);
    g[j] = (kHit && j == rel) ? (p - 1.0f) * tau : p * tau;
  }
  if (__any_sync(0xffffffffu, xmax > kTanhXmax)) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float x = __uint_as_float(r[j]) * inv_c;
      const float th = tanh_any(x);
      const float p = ex2_approx(fmaf(th, cl2e, -lse2));
      const float tau = fmaf(-th, th, 1.0f);
      g[j] = (j == rel) ? (p - 1.0f) * tau : p * tau;
    }
  }
  if (lim < 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) g[j] = (j < lim) ? g[j] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
    out[j] = *reinterpret_cast<uint32_t*>(&b);
  }
}

// DW: column = row i of the tile with lse2[i] and hit[i] (lane index of the
// target inside this vocab block, or -1) from shared memory; lane = vocab.
__device__ __forceinline__ void g_chunk_dw(const uint32_t (&r)[32], float inv_c, float cl2e, const float* lse2,
                                           const int* hit, int my_lane, uint32_t (&out)[16]) {
  float xmax = 0.f;
  float g[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float x = __uint_as_float(r[j]) * inv_c;
    xmax = fmaxf(xmax, fabsf(x));
    const float th = tanh_poly(x);
    const float p = ex2_approx(fmaf(th, cl2e, -lse2[j]));
    const float tau = fmaf(-th, th, 1.0f);
    g[j] = (hit[j] == my_lane) ? (p - 1.0f) * tau : p * tau;
  }
  if (__any_sync(0xffffffffu, xmax > kTanhXmax)) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float x = __uint_as_float(r[j]) * inv_c;
      const float th = tanh_any(x);
      const float p = ex2_approx(fmaf(th, cl2e, -lse2[j]));
      const float tau = fmaf(-th, th, 1.0f);
      g[j] = (hit[j] == my_lane) ? (p - 1.0f) * tau : p * tau;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    __nv_bfloat162 b = __floats2bfloat162_rn(g[2 * j], g[2 * j + 1]);
    out[j] = *reinterpret_cast<uint32_t*>(&b);
  }
}

// Tile range of unit u: the stationary block and the streamed tiles.
__device__ __forceinline__ void unit_range(const Params& p, int u, int& blk, int& t0, int& t1) {
  blk = u / p.split;
  const int s = u % p.split;
  t0 = static_cast<int>(static_cast<long long>(s) * p.n_tiles / p.split);
  t1 = static_cast<int>(static_cast<long long>(s + 1) * p.n_tiles / p.split);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  // Z CTA barriers
  uint64_t* zy_full = bars + 0;     // [YSTAGES]
  uint64_t* zy_empty = bars + 4;    // [YSTAGES]
  uint64_t* x_full = bars + 8;
  uint64_t* x_empty = bars + 9;
  uint64_t* acc_full = bars + 10;   // [2]  Z: z tiles; A: [0] = accumulator done
  uint64_t* acc_empty = bars + 12;  // [2]  Z: z tiles; A: [0] = accumulator drained
  uint64_t* p_empty = bars + 14;    // [2]  in Z, arrived by A's MMA commit
  // A CTA barriers
  uint64_t* p_full = bars + 16;     // [2]  in A, arrived by Z's epilogue warps
  uint64_t* ay_full = bars + 18;    // [2]  halves of the Y tile
  uint64_t* ay_empty = bars + 20;   // [2]
  uint64_t* mma_done = bars + 22;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + BAR_OFF + 196);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;
  const bool is_z = (rank == 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < YSTAGES; ++i) {
      mbar_init(zy_full + i, 1);
      mbar_init(zy_empty + i, 1);
    }
    mbar_init(x_full, 1);
    mbar_init(x_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, EPI_WARPS);
      mbar_init(p_empty + i, 1);
      mbar_init(p_full + i, EPI_WARPS);
      mbar_init(ay_full + i, 1);
      mbar_init(ay_empty + i, 1);
    }
    mbar_init(mma_done, 1);
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
        int stage = 0;
        uint32_t phase = 0, xph = 0;
        bool first = true, ok = true;
        uint32_t pend = 0, pend_ph[YSTAGES] = {0, 0, 0, 0};
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          if (!first) {
            ok = mbar_wait(x_empty, xph, abort_flag, p.status);
            xph ^= 1u;
            if (!ok) break;
          }
          first = false;
          mbar_expect_tx(x_full, p.KC * CHUNK);
          for (int kc = 0; kc < p.KC; ++kc) tma_load_2d(smem + Z_X + kc * CHUNK, &tm_x, x_full, kc * KB, blk * BM);
          for (int t = t0; t < t1 && ok; ++t) {
            for (int kc = 0; kc < p.KC; ++kc) {
              ok = mbar_wait(zy_empty + stage, phase ^ 1u, abort_flag, p.status);
              if (!ok) break;
              mbar_expect_tx(zy_full + stage, CHUNK);
              tma_load_2d(smem + Z_Y + stage * CHUNK, &tm_y, zy_full + stage, kc * KB, t * BT);
              pend |= 1u << stage;
              pend_ph[stage] = phase;
              if (++stage == YSTAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
        if (!ok) {
          const unsigned long long t0 = globaltimer_ns();
          for (int s = 0; s < YSTAGES; ++s)
            if (pend & (1u << s))
              while (!mbar_try_wait(smem_u32(zy_full + s), pend_ph[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
              }
        }
      }
    } else if (warp == MMA_WARP) {
      if (lane == 0) {
        int stage = 0, acc = 0;
        uint32_t phase = 0, aph = 0, xph = 0;
        bool ok = true;
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          ok = mbar_wait(x_full, xph, abort_flag, p.status);
          xph ^= 1u;
          if (!ok) break;
          for (int t = t0; t < t1 && ok; ++t) {
            ok = mbar_wait(acc_empty + acc, aph ^ 1u, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BT);
            for (int kc = 0; kc < p.KC; ++kc) {
              ok = mbar_wait(zy_full + stage, phase, abort_flag, p.status);
              if (!ok) break;
              tc_fence_after();
              const uint32_t xa = smem_u32(smem + Z_X + kc * CHUNK);
              const uint32_t ya = smem_u32(smem + Z_Y + stage * CHUNK);
#pragma unroll
              for (int k = 0; k < KB / 16; ++k)
                umma_bf16(d_tmem, sdesc_sw128(xa + k * 32, 16, 1024), sdesc_sw128(ya + k * 32, 16, 1024), IDESC_Z,
                          (kc | k) != 0 ? 1u : 0u);
              umma_commit(zy_empty + stage);
              if (++stage == YSTAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit(acc_full + acc);
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
          }
          if (ok) umma_commit(x_empty);
        }
        umma_commit(mma_done);
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(mma_done), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    } else {
      // ---- Z epilogue: z tile -> P tile in the peer's shared memory ----
      const int q = warp & 3;    // lanes 32q .. 32q+31
      const int hc = warp >> 2;  // columns 64hc .. 64hc+63 (one K chunk of P)
      const int m = q * 32 + lane;  // row of the P tile (= TMEM lane)
      // DW: warp-private copy of the row data of its 64 columns.
      float* side_lse = reinterpret_cast<float*>(smem + Z_SIDE) + warp * 128;
      int* side_hit = reinterpret_cast<int*>(side_lse + 64);
      const uint32_t peer_p = mapa_shared(smem_u32(smem + A_P), 1);
      const uint32_t peer_pfull = mapa_shared(smem_u32(p_full), 1);
      int acc = 0, slot = 0;
      uint32_t aph = 0, sph = 0;
      bool ok = true;
      for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
        int blk, t0, t1;
        unit_range(p, u, blk, t0, t1);
        // DH: this thread's row data.
        float lse2 = __int_as_float(0x7f800000);  // +inf: row contributes nothing
        long long trow = -1;
        if (MODE == DH) {
          const int row = blk * BM + m;
          if (row < p.N && (!p.mask || p.mask[row])) {
            const long long tt = p.tgt[row];
            lse2 = p.lse[row] * kLog2e;
            if (tt >= 0 && tt < p.V) trow = tt;
            else atomicOr(p.status, ST_EDATA);
          }
        }
        const int my_vocab_lane = m;  // DW: vocab index inside the block
        for (int t = t0; t < t1; ++t) {
          if (MODE == DW) {
            // Rows of this warp's 64 columns: lse * log2(e) and the lane
            // (vocab inside the block) of their target, or -1.
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int col = hc * 64 + k * 32 + lane;
              const int row = t * BT + col;
              float l2 = __int_as_float(0x7f800000);
              int hl = -1;
              if (row < p.N && (!p.mask || p.mask[row])) {
                const long long tt = p.tgt[row];
                l2 = p.lse[row] * kLog2e;
                if (tt < 0 || tt >= p.V) atomicOr(p.status, ST_EDATA);
                else if (tt >= static_cast<long long>(blk) * BM && tt < static_cast<long long>(blk) * BM + BM)
                  hl = static_cast<int>(tt - static_cast<long long>(blk) * BM);
              }
              side_lse[k * 32 + lane] = l2;
              side_hit[k * 32 + lane] = hl;
            }
            __syncwarp();
          }
          ok = mbar_wait(acc_full + acc, aph, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          ok = mbar_wait<true>(p_empty + slot, sph ^ 1u, abort_flag, p.status);
          if (!ok) break;
          const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BT + hc * 64);
          const uint32_t dst_row = peer_p + static_cast<uint32_t>(slot) * P_SLOT + static_cast<uint32_t>(hc) * CHUNK +
                                   static_cast<uint32_t>(m) * 128u;
#pragma unroll 1
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t r[32];
            tmem_ld32(tb + ch * 32, r);
            tmem_ld_wait();
            reg_fence32(r);
            uint32_t packed[16];
            const int c0 = hc * 64 + ch * 32;  // column inside the tile
            if (MODE == DH) {
              const int cbase = t * BT + c0;   // vocab index
              const int lim = min(32, p.V - cbase);
              const long long relw = trow - cbase;
              const int rel = (relw >= 0 && relw < 32) ? static_cast<int>(relw) : -1;
              if (__any_sync(0xffffffffu, rel >= 0))
                g_chunk_dh<true>(r, p.inv_c, p.cl2e, lse2, rel, lim, packed);
              else
                g_chunk_dh<false>(r, p.inv_c, p.cl2e, lse2, -1, lim, packed);
            } else {
              g_chunk_dw(r, p.inv_c, p.cl2e, side_lse + ch * 32, side_hit + ch * 32, my_vocab_lane, packed);
            }
            // 4 x 16-byte units of this 32-column chunk, 128B-swizzled.
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint32_t unit = static_cast<uint32_t>(ch * 4 + v);
              const uint32_t addr = dst_row + ((unit ^ static_cast<uint32_t>(m & 7)) << 4);
              st_cluster_v4(addr, packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
            }
          }
          tc_fence_before();
          fence_proxy_async_cluster();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(acc_empty + acc);
            mbar_arrive_cluster(peer_pfull + static_cast<uint32_t>(slot) * 8u);
          }
          acc ^= 1;
          if (acc == 0) aph ^= 1u;
          slot ^= 1;
          if (slot == 0) sph ^= 1u;
        }
      }
    }
  } else {
    // =========================== A CTA ===========================
    if (warp == TMA_WARP) {
      if (lane == 0) {
        uint32_t yph = 0;  // shared by both halves: each completes once per tile
        bool ok = true;
        uint32_t pend = 0, pend_ph[2] = {0, 0};
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          for (int t = t0; t < t1 && ok; ++t) {
            for (int half = 0; half < 2 && ok; ++half) {
              const int kc0 = half == 0 ? 0 : (p.KC + 1) / 2;
              const int kc1 = half == 0 ? (p.KC + 1) / 2 : p.KC;
              if (kc1 == kc0) continue;
              ok = mbar_wait(ay_empty + half, yph ^ 1u, abort_flag, p.status);
              if (!ok) break;
              mbar_expect_tx(ay_full + half, (kc1 - kc0) * CHUNK);
              for (int kc = kc0; kc < kc1; ++kc) tma_load_2d(smem + A_Y + kc * CHUNK, &tm_y, ay_full + half, kc * KB, t * BT);
              pend |= 1u << half;
              pend_ph[half] = yph;
            }
            yph ^= 1u;
          }
        }
        if (!ok) {
          const unsigned long long t0 = globaltimer_ns();
          for (int s = 0; s < 2; ++s)
            if (pend & (1u << s))
              while (!mbar_try_wait(smem_u32(ay_full + s), pend_ph[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
              }
        }
      }
    } else if (warp == MMA_WARP) {
      if (lane == 0) {
        uint32_t yph = 0, sph = 0, dph = 0;
        int slot = 0;
        bool ok = true;
        // The accumulator's d columns in two N halves of nh0 and nh1 chunks.
        const int nh0 = (p.KC + 1) / 2;
        const int nh1 = p.KC - nh0;
        for (int u = cluster; u < p.n_units && ok; u += n_clusters) {
          int blk, t0, t1;
          unit_range(p, u, blk, t0, t1);
          ok = mbar_wait(acc_empty, dph ^ 1u, abort_flag, p.status);  // accumulator drained
          dph ^= 1u;
          if (!ok) break;
          tc_fence_after();
          for (int t = t0; t < t1 && ok; ++t) {
            ok = mbar_wait<true>(p_full + slot, sph, abort_flag, p.status);
            if (!ok) break;
            tc_fence_after();
            fence_proxy_async_smem();
            const uint32_t pa = smem_u32(smem + A_P + slot * P_SLOT);
            for (int half = 0; half < 2; ++half) {
              const int nh = half == 0 ? nh0 : nh1;
              if (nh == 0) continue;
              ok = mbar_wait(ay_full + half, yph, abort_flag, p.status);
              if (!ok) break;
              tc_fence_after();
              const uint32_t idesc = idesc_bf16_f32(128, 64 * nh, false, true);
              const uint32_t yb = smem_u32(smem + A_Y + half * nh0 * CHUNK);
              const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(half * 64 * nh0);
#pragma unroll 1
              for (int ks = 0; ks < BT / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(pa + (ks >> 2) * CHUNK + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(yb + ks * 2048, CHUNK, 1024);
                umma_bf16(d_tmem, ad, bd, idesc, (t != t0 || ks != 0) ? 1u : 0u);
              }
              umma_commit(ay_empty + half);
            }
            if (!ok) break;
            umma_commit_mc(p_empty + slot, static_cast<uint16_t>(1u << 0));  // P slot free (Z CTA)
            yph ^= 1u;
            slot ^= 1;
            if (slot == 0) sph ^= 1u;
          }
          if (ok) umma_commit(acc_full);  // accumulator of this unit complete
        }
        umma_commit(mma_done);
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(mma_done), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    } else {
      // ---- A drain: accumulator -> dh / dW ----
      const int q = warp & 3;
      const int hc = warp >> 2;       // column half of the accumulator
      const int m = q * 32 + lane;
      uint32_t fph = 0;
      for (int u = cluster; u < p.n_units; u += n_clusters) {
        int blk, t0, t1;
        unit_range(p, u, blk, t0, t1);
        if (!mbar_wait(acc_full, fph, abort_flag, p.status)) break;
        fph ^= 1u;
        tc_fence_after();
        const int row = blk * BM + m;  // DH: token row; DW: vocab row
        const int ncols_half = p.d / 2;
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(hc * ncols_half);
#pragma unroll 1
        for (int ch = 0; ch < ncols_half / 32; ++ch) {
          uint32_t r[32];
          tmem_ld32(tb + ch * 32, r);
          tmem_ld_wait();
          reg_fence32(r);
          const int col = hc * ncols_half + ch * 32;
          if (MODE == DH) {
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
                const int s = u % p.split;
                float4* dst = reinterpret_cast<float4*>(
                    p.dw_part + (static_cast<long long>(s) * p.V_pad + row) * p.d + col);
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
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

// dW = (accumulate ? dW : 0) + w * sum_{s < split} part[s], in split order.
__global__ void dw_split_reduce_kernel(const float4* __restrict__ part, int split, long long V_pad_d4, long long n4,
                                       float w, int accumulate, float4* __restrict__ dW) {
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n4;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    float4 s = part[e];
    for (int k = 1; k < split; ++k) {
      const float4 v = part[static_cast<long long>(k) * V_pad_d4 + e];
      s.x += v.x;
      s.y += v.y;
      s.z += v.z;
      s.w += v.w;
    }
    float4 o = make_float4(w * s.x, w * s.y, w * s.z, w * s.w);
    if (accumulate) {
      const float4 b = dW[e];
      o.x += b.x;
      o.y += b.y;
      o.z += b.z;
      o.w += b.w;
    }
    dW[e] = o;
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

inline size_t scratch_bytes(long long N, long long V, long long d) {
  const long long nt = cdivll(N, BT);
  const long long s = nt < MAX_SPLIT ? nt : MAX_SPLIT;
  if (s <= 1) return 0;
  return static_cast<size_t>(s) * static_cast<size_t>(cdivll(V, BM) * BM) * static_cast<size_t>(d) * 4u;
}

inline int setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(bwd_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_kernel<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) {
    set_last_error(std::string("cudaFuncSetAttribute(bwd): ") + cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

// Co-resident 2-CTA clusters for this kernel (cached per process).
inline int max_clusters(int sms) {
  static int cached = 0;
  if (cached) return cached;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sms / 2));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, bwd_kernel<DH>, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = sms / 2;
  }
  cached = n;
  return n;
}

template <int MODE>
inline int launch_mode(const CUtensorMap& tx, const CUtensorMap& ty, const Params& p, int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_kernel<MODE>, tx, ty, p);
  if (e != cudaSuccess) {
    set_last_error(std::string("bwd_kernel launch: ") + cudaGetErrorString(e));
    return 3;
  }
  return 0;
}

inline int launch(const uint16_t* h, long long ldh, const uint16_t* W, long long N, long long V, long long d,
                  const int64_t* tgt, const uint8_t* mask, float c, const float* lse, float w, uint16_t* dh, float* dW,
                  int accumulate, unsigned* status, void* scratch, int sms, cudaStream_t s) {
  CUtensorMap tm_h, tm_w;
  if (int rc = make_map_bf16(&tm_h, h, d, N, ldh * 2, KB, 128); rc) return rc;
  if (int rc = make_map_bf16(&tm_w, W, d, V, d * 2, KB, 128); rc) return rc;
  const int clusters_max = max_clusters(sms);
  Params p{};
  p.N = static_cast<int>(N);
  p.V = static_cast<int>(V);
  p.d = static_cast<int>(d);
  p.KC = static_cast<int>(d / KB);
  p.tgt = tgt;
  p.mask = mask;
  p.lse = lse;
  p.inv_c = 1.0f / c;
  p.cl2e = c * kLog2e;
  p.w = w;
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
    if (int rc = launch_mode<DH>(tm_h, tm_w, q, cl, s); rc) return rc;
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
    if (int rc = launch_mode<DW>(tm_w, tm_h, q, cl, s); rc) return rc;
    if (q.split > 1) {
      const long long n4 = V * d / 4;
      const int blocks = static_cast<int>(cdivll(n4, 256) < sms * 8 ? cdivll(n4, 256) : sms * 8);
      count_launches(1);
      dw_split_reduce_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(scratch), q.split,
                                                    static_cast<long long>(q.V_pad) * d / 4, n4, w, accumulate,
                                                    reinterpret_cast<float4*>(dW));
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) {
        set_last_error(std::string("dw_split_reduce launch: ") + cudaGetErrorString(e));
        return 3;
      }
    }
  }
  return 0;
}

}  // namespace bwdk
}  // namespace lmce
