// fwd_kernel.cuh -- forward of the fused tied-LM-head + softcapped
// cross-entropy: z = h W^T on tcgen05 tensor cores into TMEM, then in the
// epilogue s = c tanh(z/c), e^s summed per row, and the target logit picked,
// so the N x V logits never leave the SM.
//
// What it computes follows the training step of the baseline
// ("parameter-golf: ... Where Model Size Becomes the Game", section "The
// Baseline Is a Map, Not the Destination": loss = criterion(logits, y)) with
// the tied head ("parameter-golf README", leaderboard row "Naive Baseline":
// TiedEmbeddings) and softcapped logits ("HYDRA Golf" stack list: "fused
// softcapped CE kernel").
//
// Design (one CTA per SM, persistent):
//  * work = tiles (row block of 128 rows) x (vocab tile of 256); CTA b takes
//    the contiguous tile range [b T / G, (b+1) T / G) in row-block-major
//    order, so a CTA keeps one h block resident across its vocab tiles.
//  * warp 8 (one lane) issues TMA: the h block (d/64 chunks of 128 x 64 bf16,
//    128B-swizzled) once per row block, W tiles in 256 x 64 chunks through a
//    3-stage ring.
//  * warp 9 (one lane) issues tcgen05.mma M=128 N=256 K=16 into one of two
//    TMEM accumulators (2 x 256 fp32 columns = all 512).
//  * warps 0-7: epilogue.  Warp w reads TMEM lanes 32 (w % 4) .. +31 (its 32
//    rows) and columns 128 (w / 4) .. +127 of the tile.  Per logit:
//    x = z / c, e = 2^(c log2(e) tanh(x)) with tanh from the minimax
//    polynomial, summed in fp32.  No running max is needed: |s| < c, so
//    S = sum e^s lies in (V e^-c, V e^c) and cannot overflow for the
//    accepted c (the host rejects c > c_max(V)).
//  * outputs per tile and half tile: the partial sum into
//    part[2 vt + half][row]; the target logit s_t into st[row] by the one
//    thread whose columns hold t.  A finalize kernel adds the partials in a
//    fixed order (deterministic) and forms lse and nll.
#pragma once
#include "ptx.cuh"
#include "softcap_math.cuh"

namespace lmce {
namespace fwdk {

constexpr int BM = 128;        // rows per block (TMEM lanes, UMMA M)
constexpr int BN = 256;        // vocab per tile (UMMA N)
constexpr int KB = 64;         // K elements per chunk (one 128-byte swizzle row)
constexpr int STAGES = 3;      // W ring depth
constexpr int MAX_KC = 8;      // d <= 512
constexpr int EPI_WARPS = 8;
constexpr int TMA_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int THREADS = 320;
constexpr uint32_t X_CHUNK = BM * KB * 2;  // 16 KB
constexpr uint32_t Y_CHUNK = BN * KB * 2;  // 32 KB
constexpr uint32_t SMEM_X = 0;
constexpr uint32_t SMEM_Y = SMEM_X + MAX_KC * X_CHUNK;
constexpr uint32_t SMEM_BAR = SMEM_Y + STAGES * Y_CHUNK;
constexpr uint32_t SMEM_BYTES = SMEM_BAR + 256 + 1024;  // + barriers + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, false);

struct Params {
  int N;                // rows addressed by the h tensor map
  const int* n_rows;    // optional device-side live row count (compacted rows)
  int V, d, KC, VT;     // vocab, model dim, d / 64, vocab tiles
  int N_pad;            // slot stride of `part`
  const int64_t* tgt;   // [N]
  float inv_c, c;
  float k[6];           // c * log2(e) * tanh polynomial coefficients
  float* part;          // [2 VT][N_pad] partial sums of e^s
  float* st;            // [N] softcapped target logit
  unsigned* status;
};

// Sum over 32 columns of 2^(c log2e tanh(z/c)); `lim` = number of valid
// columns (32 except in the last vocab tile).
__device__ __forceinline__ float chunk_sum(const uint32_t (&r)[32], const Params& p, int lim) {
  float xmax = 0.f;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    float e[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x = __uint_as_float(r[j + u]) * p.inv_c;
      xmax = fmaxf(xmax, fabsf(x));
      e[u] = ex2_approx(x * tanh_poly_scaled(x * x, p.k));
    }
    if (lim < 32) {
#pragma unroll
      for (int u = 0; u < 4; ++u) e[u] = (j + u < lim) ? e[u] : 0.f;
    }
    s0 += e[0];
    s1 += e[1];
    s2 += e[2];
    s3 += e[3];
  }
  float s = (s0 + s1) + (s2 + s3);
  // Rare path (some |x| beyond the polynomial's range): recompute the chunk
  // with the exact-form tanh for those elements.
  if (__any_sync(0xffffffffu, xmax > kTanhXmax)) {
    float a0 = 0.f, a1 = 0.f;
    const float cl2e = p.c * kLog2e;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float x0 = __uint_as_float(r[j]) * p.inv_c;
      const float x1 = __uint_as_float(r[j + 1]) * p.inv_c;
      float e0 = ex2_approx(cl2e * tanh_any(x0));
      float e1 = ex2_approx(cl2e * tanh_any(x1));
      a0 += (j < lim) ? e0 : 0.f;
      a1 += (j + 1 < lim) ? e1 : 0.f;
    }
    s = a0 + a1;
  }
  return s;
}

__global__ void __launch_bounds__(THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
               const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SMEM_BAR);
  uint64_t* y_full = bars;          // [STAGES]
  uint64_t* y_empty = bars + 3;     // [STAGES]
  uint64_t* x_full = bars + 6;
  uint64_t* x_empty = bars + 7;
  uint64_t* acc_full = bars + 8;    // [2]
  uint64_t* acc_empty = bars + 10;  // [2]
  uint64_t* mma_done = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SMEM_BAR + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SMEM_BAR + 132);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int n_rows = p.n_rows ? min(*p.n_rows, p.N) : p.N;
  const int NB = (n_rows + BM - 1) / BM;
  const long long T = static_cast<long long>(NB) * p.VT;
  const long long g_begin = static_cast<long long>(blockIdx.x) * T / gridDim.x;
  const long long g_end = static_cast<long long>(blockIdx.x + 1) * T / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(y_full + i, 1);
      mbar_init(y_empty + i, 1);
    }
    mbar_init(x_full, 1);
    mbar_init(x_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + i, 1);
      mbar_init(acc_empty + i, EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_h);
    tma_prefetch_desc(&tm_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == TMA_WARP) {
    if (lane == 0 && g_begin < g_end) {
      int stage = 0;
      uint32_t phase = 0, xph = 0;
      int prev_rb = -1;
      uint32_t pend = 0;     // stages with a load in flight that nobody waited for
      uint32_t pend_ph[STAGES] = {0, 0, 0};
      bool ok = true;
      for (long long g = g_begin; g < g_end && ok; ++g) {
        const int rb = static_cast<int>(g / p.VT);
        const int vt = static_cast<int>(g % p.VT);
        if (rb != prev_rb) {
          if (prev_rb >= 0) {
            ok = mbar_wait(x_empty, xph, abort_flag, p.status);
            xph ^= 1u;
            if (!ok) break;
          }
          mbar_expect_tx(x_full, p.KC * X_CHUNK);
          for (int kc = 0; kc < p.KC; ++kc)
            tma_load_2d(smem + SMEM_X + kc * X_CHUNK, &tm_h, x_full, kc * KB, rb * BM);
          prev_rb = rb;
        }
        for (int kc = 0; kc < p.KC; ++kc) {
          ok = mbar_wait(y_empty + stage, phase ^ 1u, abort_flag, p.status);
          if (!ok) break;
          mbar_expect_tx(y_full + stage, Y_CHUNK);
          tma_load_2d(smem + SMEM_Y + stage * Y_CHUNK, &tm_w, y_full + stage, kc * KB, vt * BN);
          pend |= 1u << stage;
          pend_ph[stage] = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every issued copy land before the CTA can exit (bounded).
        const unsigned long long t0 = globaltimer_ns();
        for (int s = 0; s < STAGES; ++s)
          if (pend & (1u << s))
            while (!mbar_try_wait(smem_u32(y_full + s), pend_ph[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0 && g_begin < g_end) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, aph = 0, xph = 0;
      int prev_rb = -1;
      bool ok = true;
      for (long long g = g_begin; g < g_end && ok; ++g) {
        const int rb = static_cast<int>(g / p.VT);
        if (rb != prev_rb) {
          ok = mbar_wait(x_full, xph, abort_flag, p.status);
          xph ^= 1u;
          if (!ok) break;
          prev_rb = rb;
        }
        ok = mbar_wait(acc_empty + acc, aph ^ 1u, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kc = 0; kc < p.KC; ++kc) {
          ok = mbar_wait(y_full + stage, phase, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t xa = smem_u32(smem + SMEM_X + kc * X_CHUNK);
          const uint32_t ya = smem_u32(smem + SMEM_Y + stage * Y_CHUNK);
#pragma unroll
          for (int k = 0; k < KB / 16; ++k) {
            umma_bf16(d_tmem, sdesc_sw128(xa + k * 32, 16, 1024), sdesc_sw128(ya + k * 32, 16, 1024), IDESC,
                      (kc | k) != 0 ? 1u : 0u);
          }
          umma_commit(y_empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(acc_full + acc);
        const bool seg_end = (g + 1 == g_end) || ((g + 1) / p.VT != rb);
        if (seg_end) umma_commit(x_empty);
        acc ^= 1;
        if (acc == 0) aph ^= 1u;
      }
      // All issued MMAs complete before TMEM is released (bounded).
      umma_commit(mma_done);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(smem_u32(mma_done), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    const int q = warp & 3;    // TMEM lane quarter -> rows 32q .. 32q+31
    const int hc = warp >> 2;  // column half of the tile
    int acc = 0;
    uint32_t aph = 0;
    int cur_rb = -1;
    int row = 0;
    long long t = -1;
    for (long long g = g_begin; g < g_end; ++g) {
      const int rb = static_cast<int>(g / p.VT);
      const int vt = static_cast<int>(g % p.VT);
      if (rb != cur_rb) {
        row = rb * BM + q * 32 + lane;
        t = (row < n_rows) ? p.tgt[row] : -1;
        cur_rb = rb;
      }
      if (!mbar_wait(acc_full + acc, aph, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN + hc * 128);
      const int col0 = vt * BN + hc * 128;
      float sum = 0.f;
      float st_val = 0.f;
      bool st_hit = false;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[32];
        tmem_ld32(tbase + ch * 32, r);
        tmem_ld_wait();
        reg_fence32(r);
        const int cbase = col0 + ch * 32;
        const int lim = min(32, p.V - cbase);
        if (lim > 0) sum += chunk_sum(r, p, lim);
        const long long rel = t - cbase;
        const bool hit = (rel >= 0 && rel < 32);
        if (__any_sync(0xffffffffu, hit)) {
          float zt = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) zt = (rel == j) ? __uint_as_float(r[j]) : zt;
          if (hit) {
            st_val = p.c * tanh_any(zt * p.inv_c);
            st_hit = true;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + acc);
      if (row < n_rows) {
        p.part[static_cast<size_t>(2 * vt + hc) * p.N_pad + row] = sum;
        if (st_hit) p.st[row] = st_val;
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace fwdk
}  // namespace lmce
