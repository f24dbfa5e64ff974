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
// rows are summed in fp32 along a fixed tree that depends only on the
// token's row count -- pieces of kPieceRows consecutive rows (in row order),
// groups of kGroupPieces consecutive pieces (in piece order), then the groups
// in order -- and the total is added into dW once.  A stable counting sort
// puts every token's rows together in row order first.
//   1. count:   per row chunk (chunk_rows(N) rows) and token, the rows
//               (chunk-major hist[c][v]), and each row's rank among the
//               chunk's rows with its id (warps walk the chunk's rows in
//               order; lanes with equal ids take consecutive ranks in lane
//               order);
//   2. tokscan: per token (one thread), the exclusive prefix of its counts
//               over the chunks (in place), its rows, pieces and groups, and
//               their exclusive scans over all tokens in one pass (256-token
//               blocks taken in ticket order publish their totals and add
//               their predecessors': decoupled look-back); each piece's
//               token recorded, the arrival counters zeroed;
//   3. place:   per row (one thread), its slot: the token's first position,
//               plus its rows in earlier chunks, plus the row's rank in its
//               chunk (stable);
//   4. pieces:  one warp per piece sums its rows (bf16 -> fp32) in row
//               order; a token with one piece adds it into dW.  Otherwise the
//               warp that completes the last piece of a group (an arrival
//               counter) sums the group's pieces in order, and the warp that
//               completes the last group of a token sums its groups in order
//               and adds the total into dW (a token with one group adds the
//               group's sum).  Which warp does a sum varies; its order does
//               not.
// The additions into dW are vector atomic adds (red.global.add.v4.f32) that
// need no read round trip.  Each dW element receives exactly one of them per
// call, so the result is that of a load, add and store, except that the
// atomic flushes a subnormal (below 2^-126 in magnitude) operand or result
// to zero.
// Rows whose id is outside [0, V) raise ST_EDATA and are skipped.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace lmce {
namespace embk {

constexpr int kPieceRows = 32;     // rows summed by one warp
constexpr int kGroupPieces = 16;   // pieces summed by one warp
constexpr int kMaxChunks = 256;    // row chunks of the counting sort
constexpr int kCountSmemV = 32768; // largest V whose chunk counts the count kernel keeps in shared memory
constexpr int kWalkers = 8;         // warps of count8_kernel walking one 1024-row chunk together
constexpr int kWalkersMaxV = 12288; // largest V whose kWalkers x V 16-bit counts fit in 192 KB of shared memory

// Rows per chunk of the counting sort for N rows (a multiple of 32).
inline long long chunk_rows(long long N) {
  long long r = 1024;
  while ((N + r - 1) / r > kMaxChunks) r *= 2;
  return r;
}
inline long long n_chunks(long long N) { return (N + chunk_rows(N) - 1) / chunk_rows(N); }
// Upper bound on the pieces: sum over tokens of ceil(count / kPieceRows).
inline long long max_pieces(long long N, long long V) {
  return (N + kPieceRows - 1) / kPieceRows + (N < V ? N : V);
}
// Upper bound on the groups of tokens with at least two pieces: such a token
// has more than kPieceRows rows, so there are fewer than N / 33 of them and
// their groups sum to less than N / 33 + (N / 32 + N / 33) / 16 < N / 16.
inline long long max_groups(long long N) { return N / 16 + 64; }

struct Layout {
  size_t hist, lrank, offs, pbase, gbase, perm, part, gpart, pcnt, gcnt, powner, lb, total;
};
// Look-back records of the token scan: per 256-token block 8 ints {flag,
// 3 block totals, 3 inclusive prefixes, unused}, then the block ticket.
inline long long lb_ints(long long V) { return 8 * ((V + 255) / 256) + 8; }
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
inline Layout layout(long long N, long long V, long long d) {
  Layout L{};
  size_t o = 0;
  L.hist = o;   // [chunks][V] int: counts, then within-token prefixes (cursors)
  o = up256(o + sizeof(int) * static_cast<size_t>(n_chunks(N)) * static_cast<size_t>(V));
  L.lrank = o;  // [N] int: rank of each row among its chunk's rows with the same id
  o = up256(o + sizeof(int) * static_cast<size_t>(N));
  L.offs = o;   // [V + 1] int: first sorted position of each token
  o = up256(o + sizeof(int) * static_cast<size_t>(V + 1));
  L.pbase = o;  // [V + 1] int: first piece of each token
  o = up256(o + sizeof(int) * static_cast<size_t>(V + 1));
  L.gbase = o;  // [V + 1] int: first group of each token (tokens with >= 2 pieces)
  o = up256(o + sizeof(int) * static_cast<size_t>(V + 1));
  L.perm = o;   // [N] int: row indices sorted by token, stable
  o = up256(o + sizeof(int) * static_cast<size_t>(N));
  L.part = o;   // [max_pieces][d] float: piece sums of tokens with several pieces
  o = up256(o + sizeof(float) * static_cast<size_t>(max_pieces(N, V)) * static_cast<size_t>(d));
  L.gpart = o;  // [max_groups][d] float: group sums of tokens with several groups
  o = up256(o + sizeof(float) * static_cast<size_t>(max_groups(N)) * static_cast<size_t>(d));
  L.pcnt = o;   // [max_groups] int: pieces of each group completed
  o = up256(o + sizeof(int) * static_cast<size_t>(max_groups(N)));
  L.gcnt = o;   // [V] int: groups of each token completed
  o = up256(o + sizeof(int) * static_cast<size_t>(V));
  L.powner = o; // [max_pieces] int: the token of each piece
  o = up256(o + sizeof(int) * static_cast<size_t>(max_pieces(N, V)));
  L.lb = o;     // look-back records and ticket of the token scan
  o = up256(o + sizeof(int) * static_cast<size_t>(lb_ints(V)));
  L.total = o;
  return L;
}

__device__ __forceinline__ bool id_ok(long long v, int V) { return v >= 0 && v < V; }

// 16 bytes of a gradient row, read once: through the non-coherent path, not
// kept in L1, with the L2 fetching 256-byte blocks (a row is 2 d bytes,
// read by the whole warp at once).  The hint took the call from 0.0459 to
// 0.0440 ms at N = 65536, d = 512.
__device__ __forceinline__ uint4 ld_row16(const uint4* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// The kernels after the first are launched with programmatic stream
// serialization: their launch overlaps the previous kernel's tail, and each
// waits here (griddepcontrol.wait) until the previous kernel has completed
// and its memory operations are visible before reading what it wrote.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The first three kernels let the next one launch its blocks at once
// (griddepcontrol.launch_dependents), so that they are resident and waiting
// in wait_prior_grid when this grid completes.
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ int ld_shared_s32(const int* p) {
  int x;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(x) : "r"(smem_u32(p)) : "memory");
  return x;
}
__device__ __forceinline__ void st_shared_s32(int* p, int x) {
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(x) : "memory");
}

// Warp-wide walk over rows i0 .. i1 - 1 of a chunk, in order, 32 at a time:
// lanes with equal ids (__match_any_sync) take consecutive ranks in lane order
// after the id's count so far, and the group's lowest lane advances the count
// in cnt (shared memory when kShared, so no access of the walk waits on a
// global store; the chunk's hist row otherwise).  The ranks are kept in
// registers and stored to lrank after each 1024 rows.
template <bool kShared>
__device__ __forceinline__ void rank_walk(const int64_t* __restrict__ ids, int i0, int i1, int V, int* cnt,
                                          int* __restrict__ lrank, unsigned* status, int lane) {
  constexpr int kSteps = 32;
  for (int b0 = i0; b0 < i1; b0 += 32 * kSteps) {
    // The chunk's ids are loaded ahead: lane l holds row b0 + 32 st + l of
    // step st (-1 for rows that do not count).
    // The status update comes after all the loads: an atomic between them
    // made each load wait for the one before it.
    int tok[kSteps], rk[kSteps];
    bool bad = false;
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const int i = b0 + 32 * st + lane;
      const long long v = i < i1 ? ids[i] : 0;
      bad |= i < i1 && !id_ok(v, V);
      tok[st] = i < i1 && id_ok(v, V) ? static_cast<int>(v) : -1;
    }
    if (bad) atomicOr(status, ST_EDATA);
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const int v = tok[st];
      const bool ok = v >= 0;
      const unsigned active = __ballot_sync(0xffffffffu, ok);
      const unsigned peers = __match_any_sync(0xffffffffu, v) & active;
      const unsigned below = peers & ((1u << lane) - 1u);
      int base = 0;
      if (ok) {
        if constexpr (kShared)
          base = ld_shared_s32(cnt + v);
        else
          base = cnt[v];
      }
      rk[st] = base + __popc(below);
      __syncwarp();
      if (ok && below == 0u) {
        if constexpr (kShared)
          st_shared_s32(cnt + v, base + __popc(peers));
        else
          cnt[v] = base + __popc(peers);
      }
      __syncwarp();
    }
#pragma unroll
    for (int st = 0; st < kSteps; ++st)
      if (tok[st] >= 0) lrank[b0 + 32 * st + lane] = rk[st];
  }
}

// 1. hist[c][v] = rows of chunk c with id v, and lrank[i] = the rank of row
//    i among the chunk's rows with the same id (the number of earlier rows
//    of the chunk with that id), by one warp's walk (rank_walk).  With
//    use_smem (V <= kCountSmemV; dynamic shared memory of V ints) the counts
//    live in shared memory and the block writes its row out whole;
//    otherwise they live in the block's hist row.  Also zeroes the token
//    scan's look-back records.
__global__ void count_kernel(const int64_t* __restrict__ ids, int N, int V, int R, int* __restrict__ hist,
                             int* __restrict__ lrank, unsigned* status, int use_smem, int* __restrict__ lb,
                             int lb_n) {
  extern __shared__ int s_hist[];
  allow_next_grid();
  // The token scan's look-back records and ticket start at zero.
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < lb_n; k += gridDim.x * blockDim.x) lb[k] = 0;
  const int c = blockIdx.x;
  const int i0 = c * R, i1 = min(N, i0 + R);
  int* h = hist + static_cast<size_t>(c) * V;
  int* cnt = use_smem ? s_hist : h;
  for (int v = threadIdx.x; v < V; v += blockDim.x) cnt[v] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    if (use_smem)
      rank_walk<true>(ids, i0, i1, V, s_hist, lrank, status, threadIdx.x);
    else
      rank_walk<false>(ids, i0, i1, V, h, lrank, status, threadIdx.x);
  }
  if (!use_smem) return;
  __syncthreads();
  for (int v = threadIdx.x; v < V; v += blockDim.x) h[v] = s_hist[v];
}

// 1b. count_kernel's results for 1024-row chunks and V <= kWalkersMaxV, with
//     the walk split over the block's 8 warps: warp w walks rows 128 w ..
//     128 w + 127 of the chunk (as rank_walk) with 16-bit counts of its own
//     (dynamic shared memory, [kWalkers][V]).  A row's rank is its rank among
//     its warp's rows with the same id plus that id's counts in the warps
//     before; the chunk's count of an id is the sum over the warps.
__global__ void __launch_bounds__(256) count8_kernel(const int64_t* __restrict__ ids, int N, int V,
                                                     int* __restrict__ hist, int* __restrict__ lrank,
                                                     unsigned* status, int* __restrict__ lb, int lb_n) {
  extern __shared__ __align__(16) uint16_t s_cnt[];
  allow_next_grid();
  // The token scan's look-back records and ticket start at zero.
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < lb_n; k += gridDim.x * blockDim.x) lb[k] = 0;
  const int c = blockIdx.x;
  const int i0 = c * 1024, i1 = min(N, i0 + 1024);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(s_cnt);
  for (int k = threadIdx.x; k < kWalkers * V / 2; k += blockDim.x) s_words[k] = 0u;
  constexpr int kSteps = 1024 / (32 * kWalkers);
  int tok[kSteps], rk[kSteps];
  bool bad = false;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int i = i0 + 32 * (kSteps * warp + st) + lane;
    const long long v = i < i1 ? ids[i] : 0;
    bad |= i < i1 && !id_ok(v, V);
    tok[st] = i < i1 && id_ok(v, V) ? static_cast<int>(v) : -1;
  }
  if (bad) atomicOr(status, ST_EDATA);
  __syncthreads();
  uint16_t* mine = s_cnt + static_cast<size_t>(warp) * V;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int v = tok[st];
    const bool ok = v >= 0;
    const unsigned active = __ballot_sync(0xffffffffu, ok);
    const unsigned peers = __match_any_sync(0xffffffffu, v) & active;
    const unsigned below = peers & ((1u << lane) - 1u);
    const int base = ok ? static_cast<int>(mine[v]) : 0;
    rk[st] = base + __popc(below);
    __syncwarp();
    if (ok && below == 0u) mine[v] = static_cast<uint16_t>(base + __popc(peers));
    __syncwarp();
  }
  __syncthreads();
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int v = tok[st];
    if (v < 0) continue;
    int b = rk[st];
    for (int w2 = 0; w2 < warp; ++w2) b += s_cnt[static_cast<size_t>(w2) * V + v];
    lrank[i0 + 32 * (kSteps * warp + st) + lane] = b;
  }
  int* h = hist + static_cast<size_t>(c) * V;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    int sum = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWalkers; ++w2) sum += s_cnt[static_cast<size_t>(w2) * V + v];
    h[v] = sum;
  }
}

// Block-wide exclusive scans (blockDim.x == 256) of three values per thread
// at once: x[k] <- the thread's prefix of value k, total[k] <- the block's sum.
__device__ __forceinline__ void block_scan3_256(int (&x)[3], int* s_warp, int (&total)[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    inc[k] = x[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += y;
    }
    if (lane == 31) s_warp[8 * k + warp] = inc[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      int w = lane < 8 ? s_warp[8 * k + lane] : 0;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < 8) s_warp[8 * k + lane] = w;  // inclusive over the warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    x[k] = (warp > 0 ? s_warp[8 * k + warp - 1] : 0) + inc[k] - x[k];
    total[k] = s_warp[8 * k + 7];
  }
}

// 2. Per token v (one thread of 256-thread blocks): hist[c][v] <- rows of v
//    in chunks before c (in place); the rows, pieces and groups of v (only
//    tokens with >= 2 pieces have groups) and their exclusive scans over all
//    tokens into offs / pbase / gbase (totals at V).  The scan is one pass:
//    blocks take tickets in start order, scan their 256 tokens, publish
//    their totals (flag 1), then add the totals of the blocks before them
//    (one warp reads 32 of them at a time), back to the nearest one that has
//    published its inclusive prefix (flag 2), and publish their own.  A
//    block only waits for blocks with lower tickets, which have started, so
//    every wait ends; each is bounded all the same (ST_ETIMEOUT).  Then
//    each piece records its token and the arrival counters of the token and
//    its groups are zeroed.
__global__ void __launch_bounds__(256) tokscan_kernel(int* __restrict__ hist, int C, int V, int* __restrict__ offs,
                                                      int* __restrict__ pbase, int* __restrict__ gbase,
                                                      int* __restrict__ gcnt, int* __restrict__ pcnt,
                                                      int* __restrict__ powner, int* lb, unsigned* status) {
  allow_next_grid();
  wait_prior_grid();
  __shared__ int s_warp[24];
  __shared__ int s_b, s_ex[3];
  const int nb = gridDim.x;
  if (threadIdx.x == 0) s_b = atomicAdd(lb + 8 * nb, 1);
  __syncthreads();
  const int b = s_b;
  const int v = b * 256 + threadIdx.x;
  int run = 0;
  if (v < V) {
    for (int c0 = 0; c0 < C; c0 += 16) {
      int x[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) x[k] = c0 + k < C ? hist[static_cast<size_t>(c0 + k) * V + v] : 0;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        if (c0 + k < C) hist[static_cast<size_t>(c0 + k) * V + v] = run;
        run += x[k];
      }
    }
  }
  const int np = (run + kPieceRows - 1) / kPieceRows;
  const int ng = np >= 2 ? (np + kGroupPieces - 1) / kGroupPieces : 0;
  int t[3];
  int pre[3] = {run, np, ng};
  block_scan3_256(pre, s_warp, t);
  const int la = pre[0], lpb = pre[1], lgb = pre[2];
  if (threadIdx.x < 32) {
    // Warp 0: publish this block's totals, then read up to 32 predecessors'
    // records at once (lane k: block b - 1 - k - 32 r), adding their totals
    // down to the nearest one that holds its inclusive prefix.
    const int lane = threadIdx.x;
    volatile int* rec = lb + 8 * b;
    int ex[3] = {0, 0, 0};
    if (b > 0) {
      if (lane == 0) {
        for (int k = 0; k < 3; ++k) rec[1 + k] = t[k];
        __threadfence();
        atomicExch(lb + 8 * b, 1);
      }
      __syncwarp();
      const long long c0 = clock64();
      int j_hi = b - 1;
      for (;;) {
        const int j = j_hi - lane;
        const volatile int* pr = lb + 8 * (j >= 0 ? j : 0);
        const int f = j >= 0 ? pr[0] : 2;  // before block 0: an inclusive prefix of 0
        const unsigned inc_mask = __ballot_sync(0xffffffffu, f == 2);
        const unsigned zero_mask = __ballot_sync(0xffffffffu, f == 0);
        const int first_inc = inc_mask ? __ffs(inc_mask) - 1 : 32;
        const unsigned need = first_inc >= 31 ? 0xffffffffu : ((2u << first_inc) - 1u);
        if (zero_mask & need) {
          if (clock64() - c0 > kWaitLimitCycles) {
            if (lane == 0) atomicOr(status, ST_ETIMEOUT);
            break;
          }
          continue;
        }
        __threadfence();
        int x[3] = {0, 0, 0};
        if (j >= 0 && lane <= first_inc) {
          const int off = lane == first_inc ? 4 : 1;
          for (int k = 0; k < 3; ++k) x[k] = pr[off + k];
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x[k] += __shfl_xor_sync(0xffffffffu, x[k], o);
          ex[k] += x[k];
        }
        if (first_inc < 32) break;
        j_hi -= 32;
      }
    }
    if (lane == 0) {
      for (int k = 0; k < 3; ++k) rec[4 + k] = ex[k] + t[k];
      __threadfence();
      atomicExch(lb + 8 * b, 2);
      for (int k = 0; k < 3; ++k) s_ex[k] = ex[k];
      if (b == nb - 1) {
        offs[V] = ex[0] + t[0];
        pbase[V] = ex[1] + t[1];
        gbase[V] = ex[2] + t[2];
      }
    }
  }
  __syncthreads();
  if (v < V) {
    offs[v] = s_ex[0] + la;
    const int pb = s_ex[1] + lpb;
    const int gb = s_ex[2] + lgb;
    pbase[v] = pb;
    gbase[v] = gb;
    gcnt[v] = 0;
    for (int p = pb; p < pb + np; ++p) powner[p] = v;
    for (int q = gb; q < gb + ng; ++q) pcnt[q] = 0;
  }
}

// 3. Row i (one thread): its slot offs[v] + hist[c][v] (the rows of v in
//    chunks before its chunk c, after the token scan) + lrank[i] gets the
//    row index (perm), so each token's rows keep their row order (stable).
//    The ids are the caller's input, which no kernel of this call writes, so
//    they are read before the wait.
__global__ void __launch_bounds__(256) place_kernel(const int64_t* __restrict__ ids, int N, int V, int R,
                                                    const int* __restrict__ hist, const int* __restrict__ lrank,
                                                    const int* __restrict__ offs, int* __restrict__ perm) {
  allow_next_grid();
  const int i = blockIdx.x * 256 + threadIdx.x;
  const long long id = i < N ? ids[i] : -1;
  wait_prior_grid();
  if (!id_ok(id, V)) return;
  const int v = static_cast<int>(id);
  perm[offs[v] + hist[static_cast<size_t>(i / R) * V + v] + lrank[i]] = i;
}

// Token owning entry p of a sorted exclusive-prefix array base[0..V]: the
// last v with base[v] <= p.
__device__ __forceinline__ int owner_of(const int* __restrict__ base, int V, int p) {
  int lo = 0, hi = V - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= p) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// dW[v][:] += s (lane l holds the float4 groups l, l + 32, l + 64, l + 96),
// by vector atomic adds.
__device__ __forceinline__ void add_row_f4(float* __restrict__ dW, int v, int ng4, const float4 (&s)[4], int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = lane + 32 * q;
    if (j < ng4) {
      float4* o = reinterpret_cast<float4*>(dW + static_cast<size_t>(v) * (4 * ng4)) + j;
      atomicAdd(o, s[q]);
    }
  }
}

// Sum, in order, of n rows of d floats starting at src (row stride d) into s
// (lane l: float4 groups l + 32 q); up to kSumBatch rows' loads in flight.
// The rows were written by other warps of the same kernel (see
// pieces_kernel), so the loads bypass L1 (ld.global.cg).
constexpr int kSumBatch = 4;
__device__ __forceinline__ void sum_rows_f4(const float* __restrict__ src, int n, int ng4, float4 (&s)[4], int lane) {
#pragma unroll
  for (int q = 0; q < 4; ++q) s[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = 0; r0 < n; r0 += kSumBatch) {
    float4 buf[kSumBatch][4];
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = lane + 32 * q;
        buf[b][q] = (r0 + b < n && j < ng4)
                        ? __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(r0 + b) * (4 * ng4)) + j)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int b = 0; b < kSumBatch; ++b) {
      if (r0 + b >= n) break;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        s[q].x += buf[b][q].x;
        s[q].y += buf[b][q].y;
        s[q].z += buf[b][q].z;
        s[q].w += buf[b][q].w;
      }
    }
  }
}

// Lane 0 adds 1 to *counter after this warp's stores are visible GPU-wide;
// returns (to every lane) whether this warp brought it to `last_value`.
__device__ __forceinline__ bool arrive_last(int* counter, int last_value, int lane) {
  __threadfence();
  __syncwarp();
  int old = 0;
  if (lane == 0) old = atomicAdd(counter, 1);
  old = __shfl_sync(0xffffffffu, old, 0);
  const bool last = old == last_value;
  if (last) __threadfence();  // the other warps' sums are read after this
  return last;
}

// 4. Piece p (one warp): the sum, in row order, of its rows of g (bf16 ->
//    fp32).  Lane l holds dims 8 l .. 8 l + 7 and 256 + 8 l .. + 7; eight
//    rows' loads are in flight at once, the additions stay in row order.  A
//    token with a single piece adds it into dW.  Otherwise part[p] = sum, and
//    the warp completing the last piece of group q (pcnt[q]) sums the
//    group's pieces in order; a token with one group adds that into dW, else
//    gpart[q] = sum and the warp completing the token's last group (gcnt[v])
//    sums its groups in order and adds the total into dW.
constexpr int kRowBatch = 8;
__global__ void __launch_bounds__(256, 2) pieces_kernel(const uint16_t* __restrict__ g, long long ldg, int d, int V,
                              const int* __restrict__ offs, const int* __restrict__ pbase,
                              const int* __restrict__ gbase, const int* __restrict__ powner,
                              const int* __restrict__ perm, float* __restrict__ part,
                              float* __restrict__ gpart, int* __restrict__ pcnt, int* __restrict__ gcnt,
                              float* __restrict__ dW) {
  wait_prior_grid();
  const int warps = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const int np = pbase[V];
  const int ng = d / 8;  // 8-dim groups of a row
  const int ng4 = d / 4;
  for (int p = blockIdx.x * warps + (threadIdx.x >> 5); p < np; p += gridDim.x * warps) {
    const int v = powner[p];
    const int start = offs[v] + (p - pbase[v]) * kPieceRows;
    const int len = min(kPieceRows, offs[v + 1] - start);
    float acc[2][8];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[q][k] = 0.f;
    for (int r0 = 0; r0 < len; r0 += kRowBatch) {
      uint4 buf[kRowBatch][2];
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        const bool live = r0 + b < len;
        const uint16_t* row = g + static_cast<long long>(live ? perm[start + r0 + b] : 0) * ldg;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int j = lane + 32 * q;
          buf[b][q] = (live && j < ng) ? ld_row16(reinterpret_cast<const uint4*>(row) + j) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int b = 0; b < kRowBatch; ++b) {
        if (r0 + b >= len) break;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t w[4] = {buf[b][q].x, buf[b][q].y, buf[b][q].z, buf[b][q].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[q][2 * k] += __uint_as_float(w[k] << 16);
            acc[q][2 * k + 1] += __uint_as_float(w[k] & 0xffff0000u);
          }
        }
      }
    }
    const int npc = pbase[v + 1] - pbase[v];
    const bool single = npc == 1;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = lane + 32 * q;
      if (j >= ng) continue;
      const float4 lo = make_float4(acc[q][0], acc[q][1], acc[q][2], acc[q][3]);
      const float4 hi = make_float4(acc[q][4], acc[q][5], acc[q][6], acc[q][7]);
      float4* o = reinterpret_cast<float4*>((single ? dW + static_cast<size_t>(v) * d : part + static_cast<size_t>(p) * d) +
                                            8 * j);
      if (single) {
        atomicAdd(o, lo);
        atomicAdd(o + 1, hi);
      } else {
        o[0] = lo;
        o[1] = hi;
      }
    }
    if (single) continue;
    // ---- the group of this piece ----
    const int gl = (p - pbase[v]) / kGroupPieces;  // group index within the token
    const int q = gbase[v] + gl;
    const int p0 = pbase[v] + gl * kGroupPieces;
    const int n_in = min(kGroupPieces, pbase[v + 1] - p0);
    if (!arrive_last(pcnt + q, n_in - 1, lane)) continue;
    float4 sg[4];
    sum_rows_f4(part + static_cast<size_t>(p0) * d, n_in, ng4, sg, lane);
    const int ngr = gbase[v + 1] - gbase[v];
    if (ngr == 1) {
      add_row_f4(dW, v, ng4, sg, lane);
      continue;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      if (j < ng4) reinterpret_cast<float4*>(gpart + static_cast<size_t>(q) * d)[j] = sg[k];
    }
    // ---- the token's groups ----
    if (!arrive_last(gcnt + v, ngr - 1, lane)) continue;
    float4 st[4];
    sum_rows_f4(gpart + static_cast<size_t>(gbase[v]) * d, ngr, ng4, st, lane);
    add_row_f4(dW, v, ng4, st, lane);
  }
}

}  // namespace embk
}  // namespace lmce
