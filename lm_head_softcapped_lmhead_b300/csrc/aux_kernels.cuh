// aux_kernels.cuh -- the small, bandwidth-bound kernels around the tensor-core
// kernels: forward finalize (lse, nll), bits-per-byte reduction, row-mask
// compaction and gather, and the per-group int4 dequantisation.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "ce_math.cuh"
#include "ptx.cuh"

namespace lmce {

// ---- forward finalize ----------------------------------------------------------
// The forward's G work groups (2-CTA clusters) cover T = ceil(rows / R) * VT
// tiles (R rows per unit), group b taking [b T / G, (b+1) T / G).  Unit u
// (tiles g0 = u VT .. g0 + VT - 1) is covered by groups b_first .. b_last;
// each non-empty one wrote, per column half, its segment's sum of e^s over
// the non-target columns into part[2 s + half][row], s = max(0, start(b) -
// g0) < VT.  S_other = the sum of those, in group and half order, in fp64;
// with e^{s_t} from st[row]: lse = ln(S_other + e^{s_t}) and
// nll = log1p(S_other / e^{s_t}).  With a
// compaction map, row r of the compacted problem goes to row idx[r] of the
// outputs.  A target outside [0, V) raises ST_EDATA and gives nll = NaN.
// With nan_on_timeout, a forward whose bounded wait expired (ST_ETIMEOUT in
// the status word) gives nll = lse = NaN on every row, since its partial sums
// are incomplete.
__global__ void fwd_finalize_kernel(const float* __restrict__ part, int VT, int G, int R, int N_pad,
                                    const float* __restrict__ st, const int64_t* __restrict__ tgt,
                                    const int* __restrict__ n_rows_dev, int N, int V, const int* __restrict__ idx,
                                    float* __restrict__ nll, float* __restrict__ lse, unsigned* status,
                                    int nan_on_timeout = 0) {
  const int n = n_rows_dev ? min(*n_rows_dev, N) : N;
  const bool timed_out = nan_on_timeout && (*reinterpret_cast<volatile unsigned*>(status) & ST_ETIMEOUT);
  const long long T = static_cast<long long>((n + R - 1) / R) * VT;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const long long u = r / R;
    const long long g0 = u * VT, g1 = g0 + VT - 1;
    const long long b_first = ((g0 + 1) * G - 1) / T;
    const long long b_last = ((g1 + 1) * G - 1) / T;
    double S = 0.0;
    for (long long b = b_first; b <= b_last; ++b) {
      const long long start = b * T / G;
      if ((b + 1) * T / G == start) continue;  // a group without tiles wrote nothing
      const size_t slot = static_cast<size_t>(start > g0 ? start - g0 : 0);
      S += static_cast<double>(part[(2 * slot) * N_pad + r]);
      S += static_cast<double>(part[(2 * slot + 1) * N_pad + r]);
    }
    // S holds the non-target terms and st[r] the target's e^{s_t}:
    // nll = -ln p_t = log1p(S / e^{s_t}) keeps its relative precision as
    // p_t -> 1.  The partials are added in fp64; the logarithms are taken in
    // fp32 (a few ulp, far below the forward's tolerance, and without the
    // slow fp64 pipe).
    const int64_t t = tgt[r];
    float v, l;
    if (timed_out) {
      v = l = __int_as_float(0x7fc00000);
    } else if (t < 0 || t >= V) {
      atomicOr(status, ST_EDATA);
      v = __int_as_float(0x7fc00000);
      l = logf(static_cast<float>(S));
    } else {
      const float et = st[r];
      const float Sf = static_cast<float>(S);
      v = nll_from_sums(Sf, et);
      l = logf(static_cast<float>(S + static_cast<double>(et)));
    }
    const int o = idx ? idx[r] : r;
    nll[o] = v;
    if (lse) lse[o] = l;
  }
}

// ---- bits per byte -----------------------------------------------------------------
struct BpbPartial {
  double sum_nll;
  long long sum_bytes;
  long long n;
};

constexpr int kBpbBlocks = 256;
constexpr int kBpbThreads = 256;

// Fixed grid and fixed summation tree: the result does not depend on the GPU.
// Bytes per row: nbytes[i], or with a per-id table lut[tgt[i]] (the
// tokenizer's byte length of the scored token); a scored row whose target is
// outside [0, V) then counts nothing and raises ST_EDATA.
// Each block adds its rows in a fixed tree and stores its partial; the block
// that stores the last partial (an arrival counter in the workspace, zero
// between calls) adds the kBpbBlocks partials in a fixed tree and makes one
// ordered, non-atomic update of the caller's accumulator.  Which block does
// that varies; the order of every sum does not.
__global__ void __launch_bounds__(kBpbThreads) bpb_kernel(const float* __restrict__ nll,
                                                          const int32_t* __restrict__ nbytes,
                                                          const uint8_t* __restrict__ mask, long long N,
                                                          BpbPartial* part, BpbPartial* acc, unsigned* cnt,
                                                          const int64_t* __restrict__ tgt = nullptr,
                                                          const int32_t* __restrict__ lut = nullptr,
                                                          long long V = 0, unsigned* status = nullptr) {
  static_assert(kBpbThreads == kBpbBlocks, "the last block adds one partial per thread");
  __shared__ double s_nll[kBpbThreads];
  __shared__ long long s_b[kBpbThreads];
  __shared__ long long s_n[kBpbThreads];
  __shared__ int s_last;
  double a = 0.0;
  long long b = 0, c = 0;
  const long long stride = static_cast<long long>(kBpbBlocks) * kBpbThreads;
  // A thread's rows i0, i0 + stride, ... in that order, sixteen at a time
  // with their loads issued together.
  constexpr int kB = 16;
  for (long long i0 = static_cast<long long>(blockIdx.x) * kBpbThreads + threadIdx.x; i0 < N; i0 += kB * stride) {
    bool live[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const long long i = i0 + k * stride;
      live[k] = i < N && (!mask || mask[i]);
    }
    float nv[kB];
    int32_t nb[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const long long i = i0 + k * stride;
      nv[k] = 0.f;
      nb[k] = 0;
      if (!live[k]) continue;
      if (lut) {
        const int64_t t = tgt[i];
        if (t < 0 || t >= V) {
          atomicOr(status, ST_EDATA);
          live[k] = false;
          continue;
        }
        nb[k] = lut[t];
      } else {
        nb[k] = nbytes[i];
      }
      nv[k] = nll[i];
    }
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      if (!live[k]) continue;
      a += static_cast<double>(nv[k]);
      b += nb[k];
      c += 1;
    }
  }
  auto tree = [&]() {
    __syncthreads();
    for (int w = kBpbThreads / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) {
        s_nll[threadIdx.x] += s_nll[threadIdx.x + w];
        s_b[threadIdx.x] += s_b[threadIdx.x + w];
        s_n[threadIdx.x] += s_n[threadIdx.x + w];
      }
      __syncthreads();
    }
  };
  s_nll[threadIdx.x] = a;
  s_b[threadIdx.x] = b;
  s_n[threadIdx.x] = c;
  tree();
  if (threadIdx.x == 0) {
    part[blockIdx.x] = BpbPartial{s_nll[0], s_b[0], s_n[0]};
    __threadfence();
    s_last = atomicAdd(cnt, 1u) == static_cast<unsigned>(kBpbBlocks - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // the other blocks' partials are read after this
  const BpbPartial* pt = part + threadIdx.x;
  s_nll[threadIdx.x] = __ldcg(&pt->sum_nll);
  s_b[threadIdx.x] = __ldcg(&pt->sum_bytes);
  s_n[threadIdx.x] = __ldcg(&pt->n);
  tree();
  if (threadIdx.x == 0) {
    acc->sum_nll += s_nll[0];
    acc->sum_bytes += s_b[0];
    acc->n += s_n[0];
    *cnt = 0u;
  }
}

// ---- row-mask compaction ---------------------------------------------------------------
constexpr int kCompactThreads = 256;
constexpr int kCompactRows = 2048;  // rows per block (8 per thread)

__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kCompactThreads / 32) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kCompactThreads / 32) s_warp[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  if (total) *total = s_warp[kCompactThreads / 32 - 1];
  __syncthreads();
  return before;
}

// passes 1 and 2: scored-row count per block of kCompactRows rows (thread t
// reads rows base + 256 k + t: coalesced); the block that stores the last
// count (an arrival counter, zero between calls: the workspace's zero-fill,
// then reset here) turns the counts into exclusive offsets in block order and
// stores the grand total, the live row count of the compacted problem.
__global__ void __launch_bounds__(kCompactThreads) compact_count_kernel(const uint8_t* __restrict__ mask, int N,
                                                                        int* __restrict__ block_count,
                                                                        int* __restrict__ n_scored,
                                                                        unsigned* __restrict__ arrivals) {
  __shared__ int s_warp[kCompactThreads / 32];
  __shared__ int s_last;
  const int base = blockIdx.x * kCompactRows + threadIdx.x;
  int c = 0;
#pragma unroll
  for (int k = 0; k < kCompactRows / kCompactThreads; ++k) {
    const int i = base + k * kCompactThreads;
    if (i < N && mask[i]) ++c;
  }
  int total;
  block_exclusive_scan(c, s_warp, &total);
  if (threadIdx.x == 0) {
    block_count[blockIdx.x] = total;
    __threadfence();
    s_last = atomicAdd(arrivals, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;  // the whole block leaves together
  __threadfence();      // the other blocks' counts are read after this
  const int nblocks = static_cast<int>(gridDim.x);
  int carry = 0;
  for (int b0 = 0; b0 < nblocks; b0 += kCompactThreads) {
    const int i = b0 + threadIdx.x;
    const int v = (i < nblocks) ? __ldcg(block_count + i) : 0;
    int tot;
    const int ex = block_exclusive_scan(v, s_warp, &tot);
    if (i < nblocks) block_count[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    *n_scored = carry;
    *arrivals = 0u;
  }
}

// pass 3: scored rows get their compacted index (idx[pos] = i, targets
// gathered) in row order; masked rows get nll = 0 (and lse = 0).  The block
// takes its rows in 256-row slices (thread t: row base + 256 k + t), each
// slice's positions from a block-wide scan, so loads and stores coalesce.
__global__ void __launch_bounds__(kCompactThreads) compact_write_kernel(
    const uint8_t* __restrict__ mask, int N, const int* __restrict__ block_offset, const int64_t* __restrict__ tgt,
    int* __restrict__ idx, int64_t* __restrict__ tgt_c, float* __restrict__ nll, float* __restrict__ lse) {
  __shared__ int s_warp[kCompactThreads / 32];
  constexpr int R = kCompactRows / kCompactThreads;
  const int base = blockIdx.x * kCompactRows + threadIdx.x;
  bool m[R];
  int64_t tv[R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int i = base + k * kCompactThreads;
    m[k] = i < N && mask[i];
  }
  // The scored rows' targets are loaded before the scans (whose barriers
  // would otherwise hold each load back until the one before it returned).
#pragma unroll
  for (int k = 0; k < R; ++k) tv[k] = m[k] ? tgt[base + k * kCompactThreads] : 0;
  int pos = block_offset[blockIdx.x];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int i = base + k * kCompactThreads;
    int tot;
    const int ex = block_exclusive_scan(m[k] ? 1 : 0, s_warp, &tot);
    if (m[k]) {
      idx[pos + ex] = i;
      tgt_c[pos + ex] = tv[k];
    } else if (i < N) {
      if (nll) nll[i] = 0.f;
      if (lse) lse[i] = 0.f;
    }
    pos += tot;
  }
}

// pass 4: h_c[r, :] = h[idx[r], :] for r < n_scored (16-byte vectors, at most
// 64 per row).  A warp copies four rows at a time: their indices, then all
// their vectors' loads (non-coherent, not kept in L1, with L2 fetching
// 256-byte blocks: each row is read once, in an order that is a gather).
__device__ __forceinline__ uint4 ld_once16(const uint4* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__global__ void gather_rows_kernel(const uint4* __restrict__ h, long long ldh_vec, const int* __restrict__ idx,
                                   const int* __restrict__ n_scored, int vec_per_row, uint4* __restrict__ h_c) {
  const int n = *n_scored;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long r0 = 4 * (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)); r0 < n;
       r0 += 4 * warps) {
    int src[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) src[k] = r0 + k < n ? idx[r0 + k] : -1;
    uint4 x[4][2];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int v = lane + 32 * q;
        x[k][q] = src[k] >= 0 && v < vec_per_row ? ld_once16(h + static_cast<long long>(src[k]) * ldh_vec + v)
                                                 : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int v = lane + 32 * q;
        if (src[k] >= 0 && v < vec_per_row) h_c[(r0 + k) * vec_per_row + v] = x[k][q];
      }
  }
}

// ---- per-group int4 head -------------------------------------------------------------
// out[v, k] = bf16_rne(q[v, k] * scale[v, k / group]).  q: two's-complement
// nibbles, element 2m in the low nibble of byte m.  The fp32 product is exact
// (4 + 11 significant bits), so the only rounding is the final RNE to bf16.
// One thread: 16 elements (8 packed bytes).
__global__ void dequant_int4_kernel(const uint8_t* __restrict__ Wq, const __half* __restrict__ scales, int V, int d,
                                    int group, __nv_bfloat16* __restrict__ out) {
  const long long per_row = d / 16;
  const long long total = static_cast<long long>(V) * per_row;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long v = e / per_row;
    const int k0 = static_cast<int>(e % per_row) * 16;
    const uint2 packed = *reinterpret_cast<const uint2*>(Wq + v * (d / 2) + k0 / 2);
    const float sc = __half2float(scales[v * (d / group) + k0 / group]);
    uint32_t words[2] = {packed.x, packed.y};
    __align__(16) __nv_bfloat16 o[16];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t byte = (words[b / 4] >> (8 * (b % 4))) & 0xFFu;
      const int lo = static_cast<int>(byte & 0xFu);
      const int hi = static_cast<int>(byte >> 4);
      o[2 * b] = __float2bfloat16_rn(static_cast<float>(lo >= 8 ? lo - 16 : lo) * sc);
      o[2 * b + 1] = __float2bfloat16_rn(static_cast<float>(hi >= 8 ? hi - 16 : hi) * sc);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + v * d + k0);
    dst[0] = *reinterpret_cast<const uint4*>(&o[0]);
    dst[1] = *reinterpret_cast<const uint4*>(&o[8]);
  }
}

// ---- forward finalize with running maxima (softcap 0 or above the fixed-shift range) ----
// As fwd_finalize_kernel, but each partial is a pair (S, m) in base 2: the
// segment's non-target terms sum to S * 2^m, i.e. sum 2^{a_j - m} with
// a = s log2(e); st[row] holds the target's a_t.  With M = the largest m_k
// and a_t, A = sum_k S_k 2^{m_k - M} (fp64, in group and half order):
//   nll = log1p(A 2^{M - a_t}),  lse = ln 2 (M + log2(A + 2^{a_t - M})).
__global__ void fwd_finalize_online_kernel(const float* __restrict__ part, const float* __restrict__ partm, int VT,
                                           int G, int R, int N_pad, const float* __restrict__ st,
                                           const int64_t* __restrict__ tgt, const int* __restrict__ n_rows_dev, int N,
                                           int V, const int* __restrict__ idx, float* __restrict__ nll,
                                           float* __restrict__ lse, unsigned* status) {
  const int n = n_rows_dev ? min(*n_rows_dev, N) : N;
  const long long T = static_cast<long long>((n + R - 1) / R) * VT;
  const double kLn2 = 0.69314718055994530942;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    const long long u = r / R;
    const long long g0 = u * VT, g1 = g0 + VT - 1;
    const long long b_first = ((g0 + 1) * G - 1) / T;
    const long long b_last = ((g1 + 1) * G - 1) / T;
    const int64_t t = tgt[r];
    const bool tv = (t >= 0 && t < V);
    double M = tv ? static_cast<double>(st[r]) : -INFINITY;
    for (long long b = b_first; b <= b_last; ++b) {
      const long long start = b * T / G;
      if ((b + 1) * T / G == start) continue;
      const size_t slot = static_cast<size_t>(start > g0 ? start - g0 : 0);
      M = fmax(M, static_cast<double>(partm[(2 * slot) * N_pad + r]));
      M = fmax(M, static_cast<double>(partm[(2 * slot + 1) * N_pad + r]));
    }
    double A = 0.0;
    for (long long b = b_first; b <= b_last; ++b) {
      const long long start = b * T / G;
      if ((b + 1) * T / G == start) continue;
      const size_t slot = static_cast<size_t>(start > g0 ? start - g0 : 0);
      for (int hh = 0; hh < 2; ++hh) {
        const float S = part[(2 * slot + hh) * N_pad + r];
        const float m = partm[(2 * slot + hh) * N_pad + r];
        if (S > 0.f) A += static_cast<double>(S) * exp2(static_cast<double>(m) - M);
      }
    }
    float v, l;
    if (!tv) {
      atomicOr(status, ST_EDATA);
      v = __int_as_float(0x7fc00000);
      l = static_cast<float>(kLn2 * (M + log2(A)));
    } else {
      const double at = static_cast<double>(st[r]);
      v = static_cast<float>(log1p(A * exp2(M - at)));
      l = static_cast<float>(kLn2 * (M + log2(A + exp2(at - M))));
    }
    const int o = idx ? idx[r] : r;
    nll[o] = v;
    if (lse) lse[o] = l;
  }
}

// ---- more storage formats of the tied table ----------------------------------------
// Asymmetric per-group int4: unsigned codes q (element 2m in the low nibble
// of byte m), fp16 scale and integer zero point z per group:
// out = bf16_rne((q - z) * scale); the fp32 product is exact (5 + 11 bits).
// One thread: 16 elements.
__global__ void dequant_int4_asym_kernel(const uint8_t* __restrict__ Wq, const __half* __restrict__ scales,
                                         const uint8_t* __restrict__ zeros, int V, int d, int group,
                                         __nv_bfloat16* __restrict__ out) {
  const long long per_row = d / 16;
  const long long total = static_cast<long long>(V) * per_row;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long v = e / per_row;
    const int k0 = static_cast<int>(e % per_row) * 16;
    const uint2 packed = *reinterpret_cast<const uint2*>(Wq + v * (d / 2) + k0 / 2);
    const long long gi = v * (d / group) + k0 / group;
    const float sc = __half2float(scales[gi]);
    const int z = zeros[gi];
    uint32_t words[2] = {packed.x, packed.y};
    __align__(16) __nv_bfloat16 o[16];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t byte = (words[b / 4] >> (8 * (b % 4))) & 0xFFu;
      o[2 * b] = __float2bfloat16_rn(static_cast<float>(static_cast<int>(byte & 0xFu) - z) * sc);
      o[2 * b + 1] = __float2bfloat16_rn(static_cast<float>(static_cast<int>(byte >> 4) - z) * sc);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + v * d + k0);
    dst[0] = *reinterpret_cast<const uint4*>(&o[0]);
    dst[1] = *reinterpret_cast<const uint4*>(&o[8]);
  }
}

// int8 rows (int7 is the same storage with |q| <= 63): out = bf16_rne(q *
// scale_row); the fp32 product is exact (7 + 11 bits).  One thread: 16
// elements.
__global__ void dequant_int8_rows_kernel(const int8_t* __restrict__ q, const __half* __restrict__ scales, int V,
                                         int d, __nv_bfloat16* __restrict__ out) {
  const long long per_row = d / 16;
  const long long total = static_cast<long long>(V) * per_row;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long v = e / per_row;
    const int k0 = static_cast<int>(e % per_row) * 16;
    const int4 raw = *reinterpret_cast<const int4*>(q + v * d + k0);
    const float sc = __half2float(scales[v]);
    const int8_t* b = reinterpret_cast<const int8_t*>(&raw);
    __align__(16) __nv_bfloat16 o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = __float2bfloat16_rn(static_cast<float>(b[j]) * sc);
    uint4* dst = reinterpret_cast<uint4*>(out + v * d + k0);
    dst[0] = *reinterpret_cast<const uint4*>(&o[0]);
    dst[1] = *reinterpret_cast<const uint4*>(&o[8]);
  }
}

// fp16 table: out = bf16_rne(w) (fp16 -> fp32 is exact).  One thread: 8
// elements.
__global__ void dequant_f16_kernel(const uint4* __restrict__ w, long long n8, uint4* __restrict__ out) {
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 raw = w[e];
    const __half* hv = reinterpret_cast<const __half*>(&raw);
    __align__(16) __nv_bfloat16 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __float2bfloat16_rn(__half2float(hv[j]));
    out[e] = *reinterpret_cast<const uint4*>(o);
  }
}

// ---- RMSNorm in front of the head ------------------------------------------------
// h = bf16(g * x * rinv), rinv = 1 / sqrt(mean(x^2) + eps) in fp32 (g NULL:
// no gain).  One warp per row; lane l holds elements 8 (l + 32 j) .. +7.
constexpr int kNormWarps = 8;
__global__ void __launch_bounds__(kNormWarps * 32) rmsnorm_fwd_kernel(const __nv_bfloat16* __restrict__ x,
                                                                      long long ldx, const float* __restrict__ g,
                                                                      float eps, int N, int d,
                                                                      __nv_bfloat16* __restrict__ h, long long ldh,
                                                                      float* __restrict__ rinv) {
  const int lane = threadIdx.x & 31;
  const int nv = d / 8;  // 16-byte vectors per row (d % 64 == 0: nv % 8 == 0)
  for (int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5); row < N; row += gridDim.x * kNormWarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(row) * ldx);
    uint4 xv[2];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = lane + 32 * j;
      xv[j] = v < nv ? xr[v] : make_uint4(0u, 0u, 0u, 0u);
      const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&xv[j]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float f = __bfloat162float(b[e]);
        ss = fmaf(f, f, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
    if (lane == 0 && rinv) rinv[row] = r;
    uint4* hr = reinterpret_cast<uint4*>(h + static_cast<long long>(row) * ldh);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = lane + 32 * j;
      if (v >= nv) continue;
      const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&xv[j]);
      __align__(16) __nv_bfloat16 o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gk = g ? g[8 * v + e] : 1.0f;
        o[e] = __float2bfloat16_rn(gk * __bfloat162float(b[e]) * r);
      }
      hr[v] = *reinterpret_cast<const uint4*>(o);
    }
  }
}

// Backward of the RMSNorm, given dh = dL/dh (bf16):
//   dx = rinv (g dh) - x rinv^3 / d * sum_k g_k dh_k x_k      (bf16 out)
//   dg partial of this block: sum over its rows of dh x rinv  (fp32, row order)
// One warp per row; each block walks a fixed contiguous row range, and its
// warps' dg sums are added in warp order, so the partials do not depend on
// timing.  dg_part: [gridDim.x][d] (nullable).
__global__ void __launch_bounds__(kNormWarps * 32) rmsnorm_bwd_kernel(
    const __nv_bfloat16* __restrict__ x, long long ldx, const float* __restrict__ g, const float* __restrict__ rinv,
    const __nv_bfloat16* __restrict__ dh, long long lddh, int N, int d, __nv_bfloat16* __restrict__ dx, long long lddx,
    float* __restrict__ dg_part) {
  __shared__ float s_dg[kNormWarps][512];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nv = d / 8;
  const long long rows_per_block = (static_cast<long long>(N) + gridDim.x - 1) / gridDim.x;
  const long long r0 = blockIdx.x * rows_per_block;
  const long long r1 = min(static_cast<long long>(N), r0 + rows_per_block);
  float acc[2][8];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
  for (long long row = r0 + warp; row < r1; row += kNormWarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * ldx);
    const uint4* gr = reinterpret_cast<const uint4*>(dh + row * lddh);
    uint4 xv[2], gv[2];
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = lane + 32 * j;
      xv[j] = v < nv ? xr[v] : make_uint4(0u, 0u, 0u, 0u);
      gv[j] = v < nv ? gr[v] : make_uint4(0u, 0u, 0u, 0u);
      const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xv[j]);
      const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv[j]);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gk = (g && v < nv) ? g[8 * v + e] : 1.0f;
        dot = fmaf(gk * __bfloat162float(gb[e]), __bfloat162float(xb[e]), dot);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float r = rinv[row];
    const float c2 = r * r * r / static_cast<float>(d) * dot;
    uint4* dr = reinterpret_cast<uint4*>(dx + row * lddx);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int v = lane + 32 * j;
      if (v >= nv) continue;
      const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xv[j]);
      const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gv[j]);
      __align__(16) __nv_bfloat16 o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float gk = g ? g[8 * v + e] : 1.0f;
        const float xf = __bfloat162float(xb[e]), df = __bfloat162float(gb[e]);
        o[e] = __float2bfloat16_rn(r * gk * df - xf * c2);
        acc[j][e] = fmaf(df * xf, r, acc[j][e]);
      }
      dr[v] = *reinterpret_cast<const uint4*>(o);
    }
  }
  if (!dg_part) return;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int v = lane + 32 * j;
    if (v < nv)
#pragma unroll
      for (int e = 0; e < 8; ++e) s_dg[warp][8 * v + e] = acc[j][e];
  }
  __syncthreads();
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < kNormWarps; ++w) s += s_dg[w][k];
    dg_part[static_cast<long long>(blockIdx.x) * d + k] = s;
  }
}

// dg (+)= sum of the block partials in block order.
__global__ void rmsnorm_dg_reduce_kernel(const float* __restrict__ dg_part, int nblk, int d, int accumulate,
                                         float* __restrict__ dg) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < d; k += gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < nblk; ++b) s += dg_part[static_cast<long long>(b) * d + k];
    dg[k] = accumulate ? dg[k] + s : s;
  }
}

// ---- bounded-wait self-test ----------------------------------------------------------
// One thread waits, with the kernels' bounded wait, on an mbarrier that gets
// its arrival only if `arrive` is set; an expired wait raises ST_ETIMEOUT in
// the status word and returns, exactly as in the tensor-core kernels.
__global__ void wait_selftest_kernel(long long limit_cycles, int arrive, unsigned* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  if (arrive) mbar_arrive(&bar);
  (void)mbar_wait(&bar, 0, &abort_flag, status, limit_cycles);
}

}  // namespace lmce
