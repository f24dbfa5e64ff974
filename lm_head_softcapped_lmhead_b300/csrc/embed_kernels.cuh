// embed_kernels.cuh -- gradient of the tied table through the input
// embedding: dW[ids[i], :] += g[i, :] for every position i.
//
// With tied embeddings the table W is both the output head and the input
// embedding ("[AGENT TASK] OpenAI Parameter Golf", architecture experiments
// table, row "Tied embeddings"; "parameter-golf README", leaderboard row
// "Naive Baseline": TiedEmbeddings), so its gradient is the head's dW plus,
// for each token, the sum of the embedding gradients of the positions that
// hold it.  The ids are Zipf-distributed: one token can own 15 % of the rows.
//
// The result is deterministic (the same bits on every call): each token's
// rows are summed in row order, in fp32, in pieces of at most kPieceRows rows
// (so that a hot token's rows are summed by many warps), and the pieces of a
// token are added in order before the one addition into dW.
//   1. count:   per token and row chunk, the rows (integer atomics),
//               stored token-major (hist[v][c]);
//   2. totals:  per token (one warp), its row count and its number of pieces;
//   3. scan:    exclusive scans of the two over the tokens (one block);
//   4. bases:   per token (one warp, an exclusive scan over its chunks), where
//               each chunk's rows of it start in the sorted order;
//   5. place:   one warp per chunk walks its rows in order and writes each row
//               index at its token's next slot (a stable counting sort);
//   6. pieces:  one warp per piece sums its rows (bf16 -> fp32) in order;
//   7. combine: one warp per token adds its pieces in order, then into dW.
// Rows whose id is outside [0, V) raise ST_EDATA and are skipped.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace lmce {
namespace embk {

constexpr int kPieceRows = 64;     // rows summed by one warp
constexpr int kMaxChunks = 1024;   // row chunks of the counting sort

// Rows per chunk of the counting sort for N rows (a multiple of 32).
inline long long chunk_rows(long long N) {
  long long r = 256;
  while ((N + r - 1) / r > kMaxChunks) r *= 2;
  return r;
}
inline long long n_chunks(long long N) { return (N + chunk_rows(N) - 1) / chunk_rows(N); }
// Upper bound on the pieces: sum over tokens of ceil(count / kPieceRows).
inline long long max_pieces(long long N, long long V) {
  return (N + kPieceRows - 1) / kPieceRows + (N < V ? N : V);
}

struct Layout {
  size_t hist, offs, pbase, perm, part, total;
};
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
inline Layout layout(long long N, long long V, long long d) {
  Layout L{};
  size_t o = 0;
  L.hist = o;   // [V][chunks] int: counts, then bases, then cursors
  o = up256(o + sizeof(int) * static_cast<size_t>(n_chunks(N)) * static_cast<size_t>(V));
  L.offs = o;   // [V + 1] int: first sorted position of each token
  o = up256(o + sizeof(int) * static_cast<size_t>(V + 1));
  L.pbase = o;  // [V + 1] int: first piece of each token
  o = up256(o + sizeof(int) * static_cast<size_t>(V + 1));
  L.perm = o;   // [N] int: row indices sorted by token, stable
  o = up256(o + sizeof(int) * static_cast<size_t>(N));
  L.part = o;   // [max_pieces][d] float: piece sums
  o = up256(o + sizeof(float) * static_cast<size_t>(max_pieces(N, V)) * static_cast<size_t>(d));
  L.total = o;
  return L;
}

__device__ __forceinline__ bool id_ok(long long v, int V) { return v >= 0 && v < V; }

// 1. hist[v][c] = rows of chunk c with id v.
__global__ void count_kernel(const int64_t* __restrict__ ids, int N, int V, int R, int C, int* __restrict__ hist,
                             unsigned* status) {
  const int c = blockIdx.x;
  const int i0 = c * R, i1 = min(N, i0 + R);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const long long v = ids[i];
    if (!id_ok(v, V)) {
      atomicOr(status, ST_EDATA);
      continue;
    }
    atomicAdd(hist + static_cast<size_t>(v) * C + c, 1);
  }
}

// 2. offs[v] = rows of token v, pbase[v] = its pieces (scanned in place next);
//    one warp per token.
__global__ void totals_kernel(const int* __restrict__ hist, int C, int V, int* __restrict__ offs,
                              int* __restrict__ pbase) {
  const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
  for (int v = blockIdx.x * warps + (threadIdx.x >> 5); v < V; v += gridDim.x * warps) {
    const int* h = hist + static_cast<size_t>(v) * C;
    int t = 0;
    for (int c = lane; c < C; c += 32) t += h[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) {
      offs[v] = t;
      pbase[v] = (t + kPieceRows - 1) / kPieceRows;
    }
  }
}

// 3. Exclusive scans of offs and pbase over v (one block), the totals in
//    entry V.
__global__ void scan_kernel(int* __restrict__ offs, int* __restrict__ pbase, int V) {
  __shared__ int s_a[1024], s_b[1024];
  __shared__ int carry_a, carry_b;
  if (threadIdx.x == 0) {
    carry_a = 0;
    carry_b = 0;
  }
  __syncthreads();
  for (int base = 0; base < V; base += blockDim.x) {
    const int v = base + threadIdx.x;
    const int a = v < V ? offs[v] : 0, b = v < V ? pbase[v] : 0;
    s_a[threadIdx.x] = a;
    s_b[threadIdx.x] = b;
    __syncthreads();
    // Hillis-Steele inclusive scan of the tile.
    for (int off = 1; off < static_cast<int>(blockDim.x); off <<= 1) {
      const int xa = threadIdx.x >= static_cast<unsigned>(off) ? s_a[threadIdx.x - off] : 0;
      const int xb = threadIdx.x >= static_cast<unsigned>(off) ? s_b[threadIdx.x - off] : 0;
      __syncthreads();
      s_a[threadIdx.x] += xa;
      s_b[threadIdx.x] += xb;
      __syncthreads();
    }
    if (v < V) {
      offs[v] = carry_a + s_a[threadIdx.x] - a;
      pbase[v] = carry_b + s_b[threadIdx.x] - b;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      carry_a += s_a[threadIdx.x];
      carry_b += s_b[threadIdx.x];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    offs[V] = carry_a;
    pbase[V] = carry_b;
  }
}

// 4. hist[v][c] <- offs[v] + rows of token v in chunks before c; one warp
//    per token, 32 chunks at a time (warp exclusive scan plus a carry).
__global__ void bases_kernel(int* __restrict__ hist, int C, int V, const int* __restrict__ offs) {
  const int warps = blockDim.x >> 5, lane = threadIdx.x & 31;
  for (int v = blockIdx.x * warps + (threadIdx.x >> 5); v < V; v += gridDim.x * warps) {
    int* h = hist + static_cast<size_t>(v) * C;
    int run = offs[v];
    for (int c0 = 0; c0 < C; c0 += 32) {
      const int c = c0 + lane;
      const int n = c < C ? h[c] : 0;
      int x = n;  // inclusive scan over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c < C) h[c] = run + x - n;
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
}

// 5. One warp per chunk, rows in order, 32 at a time: lanes with equal ids
//    take consecutive slots in lane order, so each token's rows keep their
//    row order (stable).
__global__ void place_kernel(const int64_t* __restrict__ ids, int N, int V, int R, int C, int* __restrict__ hist,
                             int* __restrict__ perm) {
  const int warps = blockDim.x >> 5;
  const int c = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (c >= C) return;
  const int i0 = c * R, i1 = min(N, i0 + R);
  int* hc = hist + c;  // hc[v * C]: this chunk's cursor of token v
  for (int b = i0; b < i1; b += 32) {
    const int i = b + lane;
    const long long v = i < i1 ? ids[i] : -1;
    const bool ok = i < i1 && id_ok(v, V);
    const unsigned active = __ballot_sync(0xffffffffu, ok);
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? v : -1ll) & active;
    int slot = 0;
    if (ok) {
      const unsigned below = peers & ((1u << lane) - 1u);
      slot = hc[static_cast<size_t>(v) * C] + __popc(below);
      perm[slot] = i;
    }
    __syncwarp();
    if (ok && (peers & ((1u << lane) - 1u)) == 0u)  // the group's lowest lane
      hc[static_cast<size_t>(v) * C] += __popc(peers);
    __syncwarp();
  }
}

// Token owning piece p: the last v with pbase[v] <= p (pbase is sorted).
__device__ __forceinline__ int piece_owner(const int* __restrict__ pbase, int V, int p) {
  int lo = 0, hi = V - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pbase[mid] <= p) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 6. part[p][:] = sum, in row order, of the rows of piece p (one warp; lane l
//    holds dims 8 l .. 8 l + 7 and 256 + 8 l .. + 7).
__global__ void pieces_kernel(const uint16_t* __restrict__ g, long long ldg, int d, int V,
                              const int* __restrict__ offs, const int* __restrict__ pbase,
                              const int* __restrict__ perm, float* __restrict__ part) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int np = pbase[V];
  const int ng = d / 8;  // 8-dim groups of a row
  for (int p = blockIdx.x * warps + (threadIdx.x >> 5); p < np; p += gridDim.x * warps) {
    const int v = piece_owner(pbase, V, p);
    const int start = offs[v] + (p - pbase[v]) * kPieceRows;
    const int len = min(kPieceRows, offs[v + 1] - start);
    float acc[2][8];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[q][k] = 0.f;
    // Loads of several rows are in flight; the additions stay in row order.
#pragma unroll 4
    for (int r = 0; r < len; ++r) {
      const uint16_t* row = g + static_cast<long long>(perm[start + r]) * ldg;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = lane + 32 * q;
        if (j < ng) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(row) + j);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[q][2 * k] += __uint_as_float(w[k] << 16);
            acc[q][2 * k + 1] += __uint_as_float(w[k] & 0xffff0000u);
          }
        }
      }
    }
    float* out = part + static_cast<size_t>(p) * d;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = lane + 32 * q;
      if (j < ng) {
        float4* o = reinterpret_cast<float4*>(out + 8 * j);
        o[0] = make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
        o[1] = make_float4(acc[q][4], acc[q][5], acc[q][6], acc[q][7]);
      }
    }
  }
}

// 7. dW[v][:] += sum of token v's pieces, in piece order (one warp per token;
//    lane l holds the float4 groups l, l + 32, l + 64, l + 96 of a row).  The
//    loads of several pieces are in flight at once; each element's additions
//    stay in piece order.
__global__ void combine_kernel(const float* __restrict__ part, const int* __restrict__ pbase, int V, int d,
                               float* __restrict__ dW) {
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ng = d / 4;  // float4 groups of a row (at most 128)
  for (int v = blockIdx.x * warps + (threadIdx.x >> 5); v < V; v += gridDim.x * warps) {
    const int p0 = pbase[v], p1 = pbase[v + 1];
    if (p0 == p1) continue;
    float4 s[4];
    const float4* b0 = reinterpret_cast<const float4*>(part + static_cast<size_t>(p0) * d);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      s[q] = j < ng ? b0[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 4
    for (int p = p0 + 1; p < p1; ++p) {
      const float4* b = reinterpret_cast<const float4*>(part + static_cast<size_t>(p) * d);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = lane + 32 * q;
        if (j < ng) {
          const float4 x = b[j];
          s[q].x += x.x;
          s[q].y += x.y;
          s[q].z += x.z;
          s[q].w += x.w;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane + 32 * q;
      if (j < ng) {
        float4* o = reinterpret_cast<float4*>(dW + static_cast<size_t>(v) * d) + j;
        float4 a = *o;
        a.x += s[q].x;
        a.y += s[q].y;
        a.z += s[q].z;
        a.w += s[q].w;
        *o = a;
      }
    }
  }
}

}  // namespace embk
}  // namespace lmce
