// aux_kernels.cuh -- the small, bandwidth-bound kernels around the tensor-core
// kernels: forward finalize (lse, nll), bits-per-byte reduction, row-mask
// compaction and gather, and the per-group int4 dequantisation.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
__global__ void fwd_finalize_kernel(const float* __restrict__ part, int VT, int G, int R, int N_pad,
                                    const float* __restrict__ st, const int64_t* __restrict__ tgt,
                                    const int* __restrict__ n_rows_dev, int N, int V, const int* __restrict__ idx,
                                    float* __restrict__ nll, float* __restrict__ lse, unsigned* status) {
  const int n = n_rows_dev ? min(*n_rows_dev, N) : N;
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
    // p_t -> 1.
    const int64_t t = tgt[r];
    float v, l;
    if (t < 0 || t >= V) {
      atomicOr(status, ST_EDATA);
      v = __int_as_float(0x7fc00000);
      l = static_cast<float>(log(S));
    } else {
      const double et = static_cast<double>(st[r]);
      v = static_cast<float>(log1p(S / et));
      l = static_cast<float>(log(S + et));
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
__global__ void __launch_bounds__(kBpbThreads) bpb_partial_kernel(const float* __restrict__ nll,
                                                                  const int32_t* __restrict__ nbytes,
                                                                  const uint8_t* __restrict__ mask, long long N,
                                                                  BpbPartial* __restrict__ out) {
  __shared__ double s_nll[kBpbThreads];
  __shared__ long long s_b[kBpbThreads];
  __shared__ long long s_n[kBpbThreads];
  double a = 0.0;
  long long b = 0, c = 0;
  const long long stride = static_cast<long long>(kBpbBlocks) * kBpbThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kBpbThreads + threadIdx.x; i < N; i += stride) {
    if (mask && !mask[i]) continue;
    a += static_cast<double>(nll[i]);
    b += nbytes[i];
    c += 1;
  }
  s_nll[threadIdx.x] = a;
  s_b[threadIdx.x] = b;
  s_n[threadIdx.x] = c;
  __syncthreads();
  for (int w = kBpbThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_nll[threadIdx.x] += s_nll[threadIdx.x + w];
      s_b[threadIdx.x] += s_b[threadIdx.x + w];
      s_n[threadIdx.x] += s_n[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) out[blockIdx.x] = BpbPartial{s_nll[0], s_b[0], s_n[0]};
}

// One block: adds the kBpbBlocks partials in a fixed tree, then adds the
// result to the caller's accumulator (one ordered, non-atomic update).
__global__ void __launch_bounds__(kBpbBlocks) bpb_final_kernel(const BpbPartial* __restrict__ part,
                                                               BpbPartial* acc) {
  __shared__ double s_nll[kBpbBlocks];
  __shared__ long long s_b[kBpbBlocks];
  __shared__ long long s_n[kBpbBlocks];
  s_nll[threadIdx.x] = part[threadIdx.x].sum_nll;
  s_b[threadIdx.x] = part[threadIdx.x].sum_bytes;
  s_n[threadIdx.x] = part[threadIdx.x].n;
  __syncthreads();
  for (int w = kBpbBlocks / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_nll[threadIdx.x] += s_nll[threadIdx.x + w];
      s_b[threadIdx.x] += s_b[threadIdx.x + w];
      s_n[threadIdx.x] += s_n[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    acc->sum_nll += s_nll[0];
    acc->sum_bytes += s_b[0];
    acc->n += s_n[0];
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

// pass 1: scored-row count per block of kCompactRows rows.
__global__ void __launch_bounds__(kCompactThreads) compact_count_kernel(const uint8_t* __restrict__ mask, int N,
                                                                        int* __restrict__ block_count) {
  __shared__ int s_warp[kCompactThreads / 32];
  const int base = blockIdx.x * kCompactRows + threadIdx.x * (kCompactRows / kCompactThreads);
  int c = 0;
  for (int k = 0; k < kCompactRows / kCompactThreads; ++k) {
    const int i = base + k;
    if (i < N && mask[i]) ++c;
  }
  int total;
  block_exclusive_scan(c, s_warp, &total);
  if (threadIdx.x == 0) block_count[blockIdx.x] = total;
}

// pass 2 (one block): exclusive scan of the block counts; the grand total is
// the live row count of the compacted problem.
__global__ void __launch_bounds__(kCompactThreads) compact_scan_kernel(int* __restrict__ block_count, int nblocks,
                                                                       int* __restrict__ n_scored) {
  __shared__ int s_warp[kCompactThreads / 32];
  int carry = 0;
  for (int base = 0; base < nblocks; base += kCompactThreads) {
    const int i = base + threadIdx.x;
    const int v = (i < nblocks) ? block_count[i] : 0;
    int total;
    const int ex = block_exclusive_scan(v, s_warp, &total);
    if (i < nblocks) block_count[i] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) *n_scored = carry;
}

// pass 3: scored rows get their compacted index (idx[pos] = i, targets
// gathered); masked rows get nll = 0 (and lse = 0).
__global__ void __launch_bounds__(kCompactThreads) compact_write_kernel(
    const uint8_t* __restrict__ mask, int N, const int* __restrict__ block_offset, const int64_t* __restrict__ tgt,
    int* __restrict__ idx, int64_t* __restrict__ tgt_c, float* __restrict__ nll, float* __restrict__ lse) {
  __shared__ int s_warp[kCompactThreads / 32];
  constexpr int R = kCompactRows / kCompactThreads;
  const int base = blockIdx.x * kCompactRows + threadIdx.x * R;
  int c = 0;
  for (int k = 0; k < R; ++k) {
    const int i = base + k;
    if (i < N && mask[i]) ++c;
  }
  int pos = block_offset[blockIdx.x] + block_exclusive_scan(c, s_warp, nullptr);
  for (int k = 0; k < R; ++k) {
    const int i = base + k;
    if (i >= N) break;
    if (mask[i]) {
      idx[pos] = i;
      tgt_c[pos] = tgt[i];
      ++pos;
    } else {
      if (nll) nll[i] = 0.f;
      if (lse) lse[i] = 0.f;
    }
  }
}

// pass 4: h_c[r, :] = h[idx[r], :] for r < n_scored (16-byte vectors).
__global__ void gather_rows_kernel(const uint4* __restrict__ h, long long ldh_vec, const int* __restrict__ idx,
                                   const int* __restrict__ n_scored, int vec_per_row, uint4* __restrict__ h_c) {
  const int n = *n_scored;
  const long long total = static_cast<long long>(n) * vec_per_row;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = e / vec_per_row;
    const int v = static_cast<int>(e % vec_per_row);
    h_c[r * vec_per_row + v] = h[static_cast<long long>(idx[r]) * ldh_vec + v];
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

}  // namespace lmce
