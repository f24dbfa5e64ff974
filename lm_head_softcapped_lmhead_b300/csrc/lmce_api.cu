// lmce_api.cu -- host side of the C ABI declared in include/lmhead_ce.h:
// argument validation (every host-detectable error returns before any
// launch), workspace layout, TMA tensor maps and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "../../include/lmhead_ce.h"
#include "aux_kernels.cuh"
#include "bwd_kernel.cuh"
#include "embed_kernels.cuh"
#include "fwd_kernel.cuh"

namespace {

thread_local std::string g_last_err;
std::atomic<unsigned long long> g_launches{0};

int cuda_fail(cudaError_t e, const char* what) {
  g_last_err = std::string(what) + ": " + cudaGetErrorString(e);
  return LMCE_ECUDA;
}

constexpr size_t kAlign = 256;
constexpr int kNormBlocks = 296;  // fixed grid of the RMSNorm backward (the gain's partial sums)
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout (byte offsets).  Every sub-buffer is 256-byte aligned.
struct Layout {
  size_t status = 0;    // unsigned status word (sticky until lmce_status)
  size_t bpb = 0;       // kBpbBlocks partials
  size_t part = 0;      // forward: [2 VT][N_pad] fp32 partial sums, then [2 VT][N_pad] running maxima
  size_t st = 0;        // forward: [N_pad] fp32 target logits
  size_t blkcnt = 0;    // masked: per-block counts / offsets
  size_t nscored = 0;   // masked: live row count
  size_t idx = 0;       // masked: [N] int32 compacted -> original row
  size_t tgt_c = 0;     // masked: [N] int64 compacted targets
  size_t h_c = 0;       // masked: [N, d] bf16 compacted rows
  size_t wdeq = 0;      // int4: [V, d] bf16 dequantised head
  size_t embed = 0;     // tied-embedding gradient: counting sort and piece sums
  size_t hn = 0;        // RMSNorm: [N, d] bf16 normalised rows
  size_t dhn = 0;       // RMSNorm: [N, d] bf16 gradient of the normalised rows
  size_t rinv = 0;      // RMSNorm: [N] fp32 reciprocal RMS
  size_t dgp = 0;       // RMSNorm: [kNormBlocks][d] fp32 partials of the gain's gradient
  size_t bwd = 0;       // backward scratch
  size_t fdrec = 0;     // forward + dh pass: per-cluster row records
  size_t total = 0;
};

Layout make_layout(int64_t N, int64_t V, int64_t d, unsigned flags) {
  Layout L;
  size_t o = 0;
  L.status = o;
  o = up(o + 64);
  L.bpb = o;
  o = up(o + sizeof(lmce::BpbPartial) * lmce::kBpbBlocks);
  const int64_t N_pad = cdiv(N, lmce::fwdk::PAIR_ROWS) * lmce::fwdk::PAIR_ROWS;
  const int64_t VT = cdiv(V, lmce::fwdk::BN);
  L.part = o;  // at most VT clusters cover one row pair: 2 VT slots per row (sums, then maxima)
  o = up(o + sizeof(float) * 2 * 2 * VT * N_pad);
  L.st = o;
  o = up(o + sizeof(float) * N_pad);
  if (flags & LMCE_WS_MASKED) {
    L.blkcnt = o;
    o = up(o + sizeof(int) * cdiv(N, lmce::kCompactRows));
    L.nscored = o;  // the live row count, then the count kernel's arrival counter
    o = up(o + 2 * sizeof(int));
    L.idx = o;
    o = up(o + sizeof(int) * N);
    L.tgt_c = o;
    o = up(o + sizeof(int64_t) * N);
    L.h_c = o;
    o = up(o + 2 * N * d);
  }
  if (flags & LMCE_WS_INT4) {
    L.wdeq = o;
    o = up(o + 2 * V * d);
  }
  if (flags & LMCE_WS_EMBED) {
    L.embed = o;
    o = up(o + lmce::embk::layout(N, V, d).total);
  }
  if (flags & LMCE_WS_RMSNORM) {
    L.dgp = o;
    o = up(o + sizeof(float) * kNormBlocks * d);
    L.rinv = o;
    o = up(o + sizeof(float) * N);
    L.hn = o;
    o = up(o + 2 * N * d);
    L.dhn = o;
    o = up(o + 2 * N * d);
  }
  L.bwd = o;
  o = up(o + lmce::bwdk::scratch_bytes(N, V, d));
  L.fdrec = o;
  o = up(o + lmce::bwdk::fd_rec_bytes(N));
  L.total = o;
  return L;
}

struct DevInfo {
  int dev = 0;
  int sms = 0;
};

// Per-device one-time set-up: SM count, architecture check, kernel
// attributes.  Thread-safe.
int dev_info(DevInfo* out) {
  static std::mutex mu;
  static bool ready[64] = {};
  static int sms[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return LMCE_ENOTSUP;
  std::lock_guard<std::mutex> lk(mu);
  if (!ready[dev]) {
    int major = 0, minor = 0, n = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3) {
      g_last_err = "device is not sm_103 (compute capability 10.3)";
      return LMCE_ENOTSUP;
    }
    if ((e = lmce::fwdk::set_attributes()) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fwd)");
    if ((e = cudaFuncSetAttribute(lmce::embk::count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sizeof(int) * lmce::embk::kCountSmemV))) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(count)");
    if ((e = cudaFuncSetAttribute(lmce::embk::count8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sizeof(uint16_t) * lmce::embk::kWalkers *
                                                   lmce::embk::kWalkersMaxV))) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(count8)");
    if (int rc = lmce::bwdk::setup_attributes(); rc != 0) return rc;
    sms[dev] = n;
    ready[dev] = true;
  }
  out->dev = dev;
  out->sms = sms[dev];
  return LMCE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

namespace lmce {

// 2-D bf16 tensor map over a row-major [outer, inner] array with row pitch
// `pitch_bytes`, box = box_inner x box_outer elements, 128-byte swizzle,
// out-of-bounds elements read as zero.
int make_map_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
                  uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_err = "cuTensorMapEncodeTiled unavailable";
    return LMCE_ECUDA;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
    return LMCE_ECUDA;
  }
  return LMCE_OK;
}

// 3-D bf16 tensor map viewing a row-major [rows, d] array (row pitch
// pitch_bytes, d a multiple of 64) as (d % 64, row, d / 64); box =
// 64 x box_rows x box_chunks, 128-byte swizzle, out-of-bounds reads as zero.
// One load of this box fills box_chunks consecutive [box_rows x 64] chunks.
int make_map_bf16_3d(CUtensorMap* m, const void* base, uint64_t d, uint64_t rows, uint64_t pitch_bytes,
                     uint32_t box_rows, uint32_t box_chunks) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_err = "cuTensorMapEncodeTiled unavailable";
    return LMCE_ECUDA;
  }
  cuuint64_t dims[3] = {64, rows, d / 64};
  cuuint64_t strides[2] = {pitch_bytes, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_err = "cuTensorMapEncodeTiled (3-D) failed with CUresult " + std::to_string(static_cast<int>(r));
    return LMCE_ECUDA;
  }
  return LMCE_OK;
}

// 2-D uint8 tensor map over a row-major [rows, inner_bytes] array (row pitch
// pitch_bytes), box = box_inner bytes x box_rows, no swizzle, out-of-bounds
// bytes read as zero.
int make_map_u8_2d(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows, uint64_t pitch_bytes,
                   uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    g_last_err = "cuTensorMapEncodeTiled unavailable";
    return LMCE_ECUDA;
  }
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_err = "cuTensorMapEncodeTiled (uint8) failed with CUresult " + std::to_string(static_cast<int>(r));
    return LMCE_ECUDA;
  }
  return LMCE_OK;
}

void set_last_error(const std::string& s) { g_last_err = s; }
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace lmce

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The one-pass forward + dh accumulates sum_j e^{s_ij} (1 - tanh^2) W_j in
// fp32 before normalising, which stays finite while V e^c max|W| < 3.4e38:
// up to c = 60 that allows |W| up to about 3e8.  Larger softcaps take the
// forward and the dh pass as two launches.
constexpr float kFusedSoftcapMax = 60.0f;

float softcap_max(int64_t V) {
  // e^{-c} must stay a normal float (c < 87.3) and V e^{c} finite (c + ln V < 88.7);
  // keep a margin of 2 on both.
  const double a = 85.0;
  const double b = 86.0 - std::log(static_cast<double>(V));
  return static_cast<float>(a < b ? a : b);
}

// Softcap c: 0 (no cap) or a finite c > 0.  Up to softcap_max(V) the
// forward sums e^s with a fixed shift; 0 and larger caps take the online
// (running-maximum) form.
bool softcap_ok(float c) { return c >= 0.0f && std::isfinite(c); }
bool softcap_online(float c, int64_t V) { return !(c > 0.0f) || c > softcap_max(V); }

// Shared shape / pointer checks of the forward and backward.
int check_common(const void* h, int64_t ldh, const void* W, int64_t N, int64_t V, int64_t d, const int64_t* tgt,
                 float softcap, void* ws) {
  if (!h || !W || !tgt || !ws) return LMCE_EINVAL;
  if (N < 1 || V < 1 || d < 1) return LMCE_EINVAL;
  if (N > (int64_t(1) << 30) || V > (int64_t(1) << 30)) return LMCE_EINVAL;
  if (d % 64 != 0 || d > 512) return LMCE_ENOTSUP;
  if (ldh < d || ldh % 8 != 0) return LMCE_EINVAL;
  if (!aligned16(h) || !aligned16(W) || !aligned16(ws)) return LMCE_EINVAL;
  if (!softcap_ok(softcap)) return LMCE_ENOTSUP;
  return LMCE_OK;
}

int bwd_launch(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
               const int64_t* tgt, const uint8_t* mask, float c, const float* lse, const float* nll, float w,
               lmce_bf16* dh, float* dW, int accumulate, unsigned* status, void* scratch, const DevInfo& di,
               cudaStream_t s) {
  return lmce::bwdk::launch(h, ldh, W, N, V, d, tgt, mask, c, lse, nll, w, dh, dW, accumulate, status, scratch,
                            di.dev, di.sms, s);
}
int fd_launch(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
              const int64_t* tgt, const uint8_t* mask, float c, float grad_scale, float* nll, float* lse,
              lmce_bf16* dh, unsigned* status, void* rec, const DevInfo& di, cudaStream_t s) {
  return lmce::bwdk::launch_fd(h, ldh, W, N, V, d, tgt, mask, c, grad_scale, nll, lse, dh, status, rec, di.dev,
                               di.sms, s);
}

// Launch with programmatic stream serialization: the kernel's launch may
// overlap the previous kernel on the stream; the kernel itself waits
// (griddepcontrol.wait) before reading what that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The one-pass forward + dh (FD) accumulates unnormalised terms: only for
// 0 < c <= kFusedSoftcapMax.
bool use_fd(float c) { return c > 0.0f && c <= kFusedSoftcapMax; }

// Forward kernel parameters for softcap c (0 = no cap: c = 1e30, where
// c tanh(z/c) equals z in fp32 and the polynomial's range check never
// triggers).
void fwd_params_softcap(lmce::fwdk::Params& p, float c) {
  const float ce = c > 0.0f ? c : 1e30f;
  p.inv_c = 1.0f / ce;
  p.c = ce;
  p.zlim2 = c > 0.0f ? (lmce::kTanhXmax * c) * (lmce::kTanhXmax * c) : HUGE_VALF;
  lmce::scaled_tanh_coeffs(static_cast<double>(ce) * 1.4426950408889634, 1.0 / static_cast<double>(ce), p.k);
}

// The forward.  With q4 (an LMCE_QHEAD_INT4 head) W is unused: the kernel's
// converter warps dequantise the packed head stage by stage (the int4 form).
int fwd_impl(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
             const int64_t* tgt, const uint8_t* mask, float c, float* nll, float* lse, void* ws, size_t ws_bytes,
             void* stream, unsigned extra_flags, const lmce_qhead* q4 = nullptr) {
  if (q4) W = static_cast<const lmce_bf16*>(q4->codes);  // only checked for alignment here
  if (int rc = check_common(h, ldh, W, N, V, d, tgt, c, ws); rc) return rc;
  if (!nll) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, (mask ? LMCE_WS_MASKED : 0u) | extra_flags);
  if (ws_bytes < L.total) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  unsigned* status = reinterpret_cast<unsigned*>(w + L.status);

  const lmce_bf16* hx = h;
  int64_t ldx = ldh;
  const int* nrows_dev = nullptr;
  const int* idx = nullptr;
  const int64_t* tg = tgt;
  if (mask) {
    const int nblk = static_cast<int>(cdiv(N, lmce::kCompactRows));
    int* blkcnt = reinterpret_cast<int*>(w + L.blkcnt);
    int* nsc = reinterpret_cast<int*>(w + L.nscored);
    int* idxp = reinterpret_cast<int*>(w + L.idx);
    int64_t* tgc = reinterpret_cast<int64_t*>(w + L.tgt_c);
    lmce_bf16* hc = reinterpret_cast<lmce_bf16*>(w + L.h_c);
    lmce::count_launches(3);
    // nsc[1] is the count kernel's arrival counter (zero between calls).
    lmce::compact_count_kernel<<<nblk, lmce::kCompactThreads, 0, s>>>(mask, static_cast<int>(N), blkcnt, nsc,
                                                                      reinterpret_cast<unsigned*>(nsc + 1));
    lmce::compact_write_kernel<<<nblk, lmce::kCompactThreads, 0, s>>>(mask, static_cast<int>(N), blkcnt, tgt, idxp,
                                                                      tgc, nll, lse);
    const int vec = static_cast<int>(d / 8);
    const int gblocks = static_cast<int>(std::min<int64_t>(cdiv(N * vec, 256), int64_t(di.sms) * 8));
    lmce::gather_rows_kernel<<<gblocks, 256, 0, s>>>(reinterpret_cast<const uint4*>(h), ldh / 8, idxp, nsc, vec,
                                                     reinterpret_cast<uint4*>(hc));
    hx = hc;
    ldx = d;
    nrows_dev = nsc;
    idx = idxp;
    tg = tgc;
  }

  CUtensorMap tm_h, tm_w;
  // h: each CTA's 128 x d rows in one load; W: 128 vocab rows x 2 chunks.
  if (int rc = lmce::make_map_bf16_3d(&tm_h, hx, d, N, ldx * 2, lmce::fwdk::BM, static_cast<uint32_t>(d / 64)); rc)
    return rc;
  if (q4) {
    if (int rc = lmce::make_map_u8_2d(&tm_w, q4->codes, d / 2, V, d / 2, lmce::fwdk::FCfg<true>::PK_ROW,
                                      lmce::fwdk::HALF_N);
        rc)
      return rc;
  } else if (int rc = lmce::make_map_bf16_3d(&tm_w, W, d, V, d * 2, lmce::fwdk::HALF_N, lmce::fwdk::SC); rc) {
    return rc;
  }

  lmce::fwdk::Params p{};
  p.N = static_cast<int>(N);
  p.n_rows = nrows_dev;
  p.V = static_cast<int>(V);
  p.d = static_cast<int>(d);
  p.KC = static_cast<int>(d / 64);
  p.VT = static_cast<int>(cdiv(V, lmce::fwdk::BN));
  p.N_pad = static_cast<int>(cdiv(N, lmce::fwdk::PAIR_ROWS) * lmce::fwdk::PAIR_ROWS);
  p.tgt = tg;
  fwd_params_softcap(p, c);
  p.part = reinterpret_cast<float*>(w + L.part);
  p.partm = p.part + static_cast<size_t>(2) * p.VT * p.N_pad;
  p.st = reinterpret_cast<float*>(w + L.st);
  p.status = status;
  p.maxseg = p.VT;
  const bool online = softcap_online(c, V);
  if (q4) {
    p.qscales = reinterpret_cast<const __half*>(q4->scales);
    p.qgroup = q4->group;
  }

  const int64_t T_max = cdiv(N, lmce::fwdk::PAIR_ROWS) * p.VT;
  const int pairs =
      static_cast<int>(std::min<int64_t>(T_max, lmce::fwdk::max_clusters(di.dev, di.sms, q4 != nullptr)));
  lmce::count_launches(2);
  if (int rc = lmce::fwdk::launch(tm_h, tm_w, p, pairs, s, online, q4 != nullptr); rc) return rc;
  cudaError_t e = cudaSuccess;
  const int fblocks = static_cast<int>(std::min<int64_t>(cdiv(N, 256), int64_t(di.sms) * 4));
  if (online)
    lmce::fwd_finalize_online_kernel<<<fblocks, 256, 0, s>>>(p.part, p.partm, p.VT, pairs, lmce::fwdk::PAIR_ROWS,
                                                             p.N_pad, p.st, tg, nrows_dev, static_cast<int>(N),
                                                             static_cast<int>(V), idx, nll, lse, status);
  else
    lmce::fwd_finalize_kernel<<<fblocks, 256, 0, s>>>(p.part, p.VT, pairs, lmce::fwdk::PAIR_ROWS, p.N_pad, p.st, tg,
                                                      nrows_dev, static_cast<int>(N), static_cast<int>(V), idx, nll,
                                                      lse, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "fwd_finalize launch");
  return LMCE_OK;
}

// Validates a quantised / fp16 head description (pointer alignment as the
// dequantisation kernels read them: 8-byte int4 code words, 16-byte int8 and
// fp16 vectors).
int check_qhead(const lmce_qhead* hd, int64_t V, int64_t d) {
  if (!hd || !hd->codes || V < 1 || d < 1 || d % 64 != 0) return LMCE_EINVAL;
  const uintptr_t q = reinterpret_cast<uintptr_t>(hd->codes);
  const uintptr_t sc = reinterpret_cast<uintptr_t>(hd->scales);
  switch (hd->format) {
    case LMCE_QHEAD_INT4:
    case LMCE_QHEAD_INT4_ASYM:
      if (!hd->scales || (q & 7u) != 0 || (sc & 1u) != 0) return LMCE_EINVAL;
      if (hd->group < 16 || hd->group % 16 != 0 || d % hd->group != 0) return LMCE_EINVAL;
      if (hd->format == LMCE_QHEAD_INT4_ASYM && !hd->zeros) return LMCE_EINVAL;
      return LMCE_OK;
    case LMCE_QHEAD_INT8_ROW:
      if (!hd->scales || (q & 15u) != 0 || (sc & 1u) != 0) return LMCE_EINVAL;
      return LMCE_OK;
    case LMCE_QHEAD_FP16:
      if ((q & 15u) != 0) return LMCE_EINVAL;
      return LMCE_OK;
    default:
      return LMCE_EINVAL;
  }
}

// out [V, d] bf16 = the dequantised head (bit-exact: one RNE rounding).
int qhead_dequant_impl(const lmce_qhead* hd, int64_t V, int64_t d, lmce_bf16* out, cudaStream_t s, int sms) {
  const int64_t per16 = V * (d / 16);
  const int blocks = static_cast<int>(std::min<int64_t>(cdiv(per16, 256), int64_t(sms) * 8));
  const auto* sc = reinterpret_cast<const __half*>(hd->scales);
  auto* o = reinterpret_cast<__nv_bfloat16*>(out);
  lmce::count_launches(1);
  switch (hd->format) {
    case LMCE_QHEAD_INT4:
      lmce::dequant_int4_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(hd->codes), sc,
                                                       static_cast<int>(V), static_cast<int>(d), hd->group, o);
      break;
    case LMCE_QHEAD_INT4_ASYM:
      lmce::dequant_int4_asym_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t*>(hd->codes), sc, hd->zeros,
                                                            static_cast<int>(V), static_cast<int>(d), hd->group, o);
      break;
    case LMCE_QHEAD_INT8_ROW:
      lmce::dequant_int8_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const int8_t*>(hd->codes), sc,
                                                            static_cast<int>(V), static_cast<int>(d), o);
      break;
    default: {
      const int64_t n8 = V * d / 8;
      const int b8 = static_cast<int>(std::min<int64_t>(cdiv(n8, 256), int64_t(sms) * 8));
      lmce::dequant_f16_kernel<<<b8, 256, 0, s>>>(static_cast<const uint4*>(hd->codes), n8,
                                                  reinterpret_cast<uint4*>(out));
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "head dequantisation launch");
  return LMCE_OK;
}

lmce_qhead int4_head(const uint8_t* Wq, const lmce_f16* scales, int group) {
  lmce_qhead hd{};
  hd.format = LMCE_QHEAD_INT4;
  hd.group = group;
  hd.codes = Wq;
  hd.scales = scales;
  hd.zeros = nullptr;
  return hd;
}

// Training step (lmhead_ce_fwd_bwd) on a workspace laid out with
// extra_flags (so that the backward's scratch does not overlap the other
// uses of the same workspace).
int fwd_bwd_impl(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                 const int64_t* tgt, const uint8_t* row_mask, float softcap, float grad_scale, float* nll, float* lse,
                 lmce_bf16* dh, float* dW, int accumulate_dW, void* ws, size_t ws_bytes, void* stream,
                 unsigned extra_flags) {
  if (int rc = check_common(h, ldh, W, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!nll || !lse) return LMCE_EINVAL;
  if (dh && !aligned16(dh)) return LMCE_EINVAL;
  if (dW && !aligned16(dW)) return LMCE_EINVAL;
  if (!std::isfinite(grad_scale)) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, (row_mask ? LMCE_WS_MASKED : 0u) | extra_flags);
  if (ws_bytes < L.total) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  char* w = static_cast<char*>(ws);
  unsigned* status = reinterpret_cast<unsigned*>(w + L.status);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dh && use_fd(softcap)) {
    // Forward and dh in one pass over the vocabulary.
    if (int rc = fd_launch(h, ldh, W, N, V, d, tgt, row_mask, softcap, grad_scale, nll, lse, dh, status,
                           w + L.fdrec, di, s);
        rc)
      return rc;
  } else {
    if (int rc = fwd_impl(h, ldh, W, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream, extra_flags);
        rc)
      return rc;
    if (dh) {
      if (int rc = bwd_launch(h, ldh, W, N, V, d, tgt, row_mask, softcap, lse, nll, grad_scale, dh, nullptr, 0,
                              status, w + L.bwd, di, s);
          rc)
        return rc;
    }
  }
  if (dW) {
    if (int rc = bwd_launch(h, ldh, W, N, V, d, tgt, row_mask, softcap, lse, nll, grad_scale, nullptr, dW,
                            accumulate_dW, status, w + L.bwd, di, s);
        rc)
      return rc;
  }
  return LMCE_OK;
}

int check_norm(const lmce_bf16* x, int64_t ldx, const float* g, int64_t N, int64_t d) {
  if (!x || N < 1 || d < 1 || N > (int64_t(1) << 30)) return LMCE_EINVAL;
  if (d % 64 != 0 || d > 512) return LMCE_ENOTSUP;
  if (ldx < d || ldx % 8 != 0 || !aligned16(x)) return LMCE_EINVAL;
  if (g && (reinterpret_cast<uintptr_t>(g) & 3u) != 0) return LMCE_EINVAL;
  return LMCE_OK;
}

int rmsnorm_fwd_impl(const lmce_bf16* x, int64_t ldx, const float* g, float eps, int64_t N, int64_t d, lmce_bf16* h,
                     int64_t ldh, float* rinv, cudaStream_t s, int sms) {
  const int blocks = static_cast<int>(std::min<int64_t>(cdiv(N, lmce::kNormWarps), int64_t(sms) * 8));
  lmce::count_launches(1);
  lmce::rmsnorm_fwd_kernel<<<blocks, lmce::kNormWarps * 32, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), ldx, g, eps, static_cast<int>(N), static_cast<int>(d),
      reinterpret_cast<__nv_bfloat16*>(h), ldh, rinv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm_fwd launch");
  return LMCE_OK;
}

int rmsnorm_bwd_impl(const lmce_bf16* x, int64_t ldx, const float* g, const float* rinv, const lmce_bf16* dh,
                     int64_t lddh, int64_t N, int64_t d, lmce_bf16* dx, int64_t lddx, float* dg, int accumulate_dg,
                     float* dgp, cudaStream_t s) {
  lmce::count_launches(dg ? 2 : 1);
  lmce::rmsnorm_bwd_kernel<<<kNormBlocks, lmce::kNormWarps * 32, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), ldx, g, rinv, reinterpret_cast<const __nv_bfloat16*>(dh), lddh,
      static_cast<int>(N), static_cast<int>(d), reinterpret_cast<__nv_bfloat16*>(dx), lddx, dg ? dgp : nullptr);
  if (dg)
    lmce::rmsnorm_dg_reduce_kernel<<<static_cast<int>(cdiv(d, 256)), 256, 0, s>>>(dgp, kNormBlocks,
                                                                                 static_cast<int>(d), accumulate_dg, dg);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm_bwd launch");
  return LMCE_OK;
}

}  // namespace

extern "C" {

size_t lmce_workspace_bytes(int64_t N, int64_t V, int64_t d, unsigned flags) {
  if (N < 1 || V < 1 || d < 1) return 0;
  return make_layout(N, V, d, flags).total;
}

float lmce_softcap_max(int64_t V) { return V < 1 ? 0.0f : softcap_max(V); }

int lmce_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 64) return LMCE_EINVAL;
  cudaError_t e = cudaMemsetAsync(ws, 0, 64, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return LMCE_OK;
}

int lmhead_ce_fwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                  const int64_t* tgt, const uint8_t* row_mask, float softcap, float* nll, float* lse, void* ws,
                  size_t ws_bytes, void* stream) {
  return fwd_impl(h, ldh, W, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream, 0u);
}

int lmhead_ce_bwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                  const int64_t* tgt, const uint8_t* row_mask, float softcap, const float* lse, const float* nll,
                  float grad_scale, lmce_bf16* dh, float* dW, int accumulate_dW, void* ws, size_t ws_bytes,
                  void* stream) {
  if (int rc = check_common(h, ldh, W, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!lse || (!dh && !dW)) return LMCE_EINVAL;
  if (dh && !aligned16(dh)) return LMCE_EINVAL;
  if (dW && !aligned16(dW)) return LMCE_EINVAL;
  if (!std::isfinite(grad_scale)) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, row_mask ? LMCE_WS_MASKED : 0u);
  if (ws_bytes < L.total) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  char* w = static_cast<char*>(ws);
  return bwd_launch(h, ldh, W, N, V, d, tgt, row_mask, softcap, lse, nll, grad_scale, dh, dW, accumulate_dW,
                    reinterpret_cast<unsigned*>(w + L.status), w + L.bwd, di, static_cast<cudaStream_t>(stream));
}

int lmhead_ce_fwd_bwd(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V, int64_t d,
                      const int64_t* tgt, const uint8_t* row_mask, float softcap, float grad_scale, float* nll,
                      float* lse, lmce_bf16* dh, float* dW, int accumulate_dW, void* ws, size_t ws_bytes,
                      void* stream) {
  return fwd_bwd_impl(h, ldh, W, N, V, d, tgt, row_mask, softcap, grad_scale, nll, lse, dh, dW, accumulate_dW, ws,
                      ws_bytes, stream, 0u);
}

int lmhead_qhead_dequant(const lmce_qhead* head, int64_t V, int64_t d, lmce_bf16* out, void* stream) {
  if (int rc = check_qhead(head, V, d); rc) return rc;
  if (!out || !aligned16(out)) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  return qhead_dequant_impl(head, V, d, out, static_cast<cudaStream_t>(stream), di.sms);
}

int lmhead_ce_fwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V, int64_t d,
                    const int64_t* tgt, const uint8_t* row_mask, float softcap, float* nll, float* lse, void* ws,
                    size_t ws_bytes, void* stream) {
  if (int rc = check_qhead(head, V, d); rc) return rc;
  if (!ws || !aligned16(ws)) return LMCE_EINVAL;
  const Layout L = make_layout(N < 1 ? 1 : N, V, d, LMCE_WS_QHEAD | (row_mask ? LMCE_WS_MASKED : 0u));
  if (ws_bytes < L.total) return LMCE_EINVAL;
  lmce_bf16* wdeq = reinterpret_cast<lmce_bf16*>(static_cast<char*>(ws) + L.wdeq);
  if (int rc = check_common(h, ldh, wdeq, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!nll) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  if (int rc = qhead_dequant_impl(head, V, d, wdeq, static_cast<cudaStream_t>(stream), di.sms); rc) return rc;
  return fwd_impl(h, ldh, wdeq, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream, LMCE_WS_QHEAD);
}

int lmhead_ce_bwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V, int64_t d,
                    const int64_t* tgt, const uint8_t* row_mask, float softcap, const float* lse, const float* nll,
                    float grad_scale, lmce_bf16* dh, void* ws, size_t ws_bytes, void* stream) {
  if (int rc = check_qhead(head, V, d); rc) return rc;
  if (!ws || !aligned16(ws) || !dh) return LMCE_EINVAL;
  const Layout L = make_layout(N < 1 ? 1 : N, V, d, LMCE_WS_QHEAD | (row_mask ? LMCE_WS_MASKED : 0u));
  if (ws_bytes < L.total) return LMCE_EINVAL;
  char* w = static_cast<char*>(ws);
  lmce_bf16* wdeq = reinterpret_cast<lmce_bf16*>(w + L.wdeq);
  if (int rc = check_common(h, ldh, wdeq, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!lse || !aligned16(dh) || !std::isfinite(grad_scale)) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = qhead_dequant_impl(head, V, d, wdeq, s, di.sms); rc) return rc;
  return bwd_launch(h, ldh, wdeq, N, V, d, tgt, row_mask, softcap, lse, nll, grad_scale, dh, nullptr, 0,
                    reinterpret_cast<unsigned*>(w + L.status), w + L.bwd, di, s);
}

int lmhead_ce_fwd_bwd_q(const lmce_bf16* h, int64_t ldh, const lmce_qhead* head, int64_t N, int64_t V, int64_t d,
                        const int64_t* tgt, const uint8_t* row_mask, float softcap, float grad_scale, float* nll,
                        float* lse, lmce_bf16* dh, void* ws, size_t ws_bytes, void* stream) {
  if (int rc = check_qhead(head, V, d); rc) return rc;
  if (!ws || !aligned16(ws)) return LMCE_EINVAL;
  const Layout L = make_layout(N < 1 ? 1 : N, V, d, LMCE_WS_QHEAD | (row_mask ? LMCE_WS_MASKED : 0u));
  if (ws_bytes < L.total) return LMCE_EINVAL;
  lmce_bf16* wdeq = reinterpret_cast<lmce_bf16*>(static_cast<char*>(ws) + L.wdeq);
  if (int rc = check_common(h, ldh, wdeq, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!nll || !lse || !dh || !aligned16(dh) || !std::isfinite(grad_scale)) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  if (int rc = qhead_dequant_impl(head, V, d, wdeq, static_cast<cudaStream_t>(stream), di.sms); rc) return rc;
  return fwd_bwd_impl(h, ldh, wdeq, N, V, d, tgt, row_mask, softcap, grad_scale, nll, lse, dh, nullptr, 0, ws,
                      ws_bytes, stream, LMCE_WS_QHEAD);
}

int lmhead_ce_fwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales, int group,
                       int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                       float* nll, float* lse, void* ws, size_t ws_bytes, void* stream) {
  const lmce_qhead hd = int4_head(Wq, scales, group);
  return lmhead_ce_fwd_q(h, ldh, &hd, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream);
}

int lmhead_ce_fwd_int4_inkernel(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales,
                                int group, int64_t N, int64_t V, int64_t d, const int64_t* tgt,
                                const uint8_t* row_mask, float softcap, float* nll, float* lse, void* ws,
                                size_t ws_bytes, void* stream) {
  const lmce_qhead hd = int4_head(Wq, scales, group);
  if (int rc = check_qhead(&hd, V, d); rc) return rc;
  if (!aligned16(Wq)) return LMCE_EINVAL;  // the packed rows are read by TMA
  return fwd_impl(h, ldh, nullptr, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream, 0u, &hd);
}

int lmhead_ce_bwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales, int group,
                       int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                       const float* lse, const float* nll, float grad_scale, lmce_bf16* dh, void* ws,
                       size_t ws_bytes, void* stream) {
  const lmce_qhead hd = int4_head(Wq, scales, group);
  return lmhead_ce_bwd_q(h, ldh, &hd, N, V, d, tgt, row_mask, softcap, lse, nll, grad_scale, dh, ws, ws_bytes,
                         stream);
}

int lmhead_ce_fwd_bwd_int4(const lmce_bf16* h, int64_t ldh, const uint8_t* Wq, const lmce_f16* scales, int group,
                           int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask,
                           float softcap, float grad_scale, float* nll, float* lse, lmce_bf16* dh, void* ws,
                           size_t ws_bytes, void* stream) {
  const lmce_qhead hd = int4_head(Wq, scales, group);
  return lmhead_ce_fwd_bwd_q(h, ldh, &hd, N, V, d, tgt, row_mask, softcap, grad_scale, nll, lse, dh, ws, ws_bytes,
                             stream);
}

int lmhead_rmsnorm_fwd(const lmce_bf16* x, int64_t ldx, const float* g, float eps, int64_t N, int64_t d,
                       lmce_bf16* h, int64_t ldh, float* rinv, void* stream) {
  if (int rc = check_norm(x, ldx, g, N, d); rc) return rc;
  if (!h || !rinv || ldh < d || ldh % 8 != 0 || !aligned16(h) || !(eps >= 0.0f) || !std::isfinite(eps))
    return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  return rmsnorm_fwd_impl(x, ldx, g, eps, N, d, h, ldh, rinv, static_cast<cudaStream_t>(stream), di.sms);
}

int lmhead_rmsnorm_bwd(const lmce_bf16* x, int64_t ldx, const float* g, const float* rinv, const lmce_bf16* dh,
                       int64_t lddh, int64_t N, int64_t d, lmce_bf16* dx, int64_t lddx, float* dg, int accumulate_dg,
                       void* ws, size_t ws_bytes, void* stream) {
  if (int rc = check_norm(x, ldx, g, N, d); rc) return rc;
  if (!rinv || !dh || !dx || lddh < d || lddh % 8 != 0 || lddx < d || lddx % 8 != 0 || !aligned16(dh) ||
      !aligned16(dx))
    return LMCE_EINVAL;
  float* dgp = nullptr;
  if (dg) {
    if (!ws || !aligned16(ws) || (reinterpret_cast<uintptr_t>(dg) & 3u) != 0) return LMCE_EINVAL;
    const Layout L = make_layout(N, 1, d, LMCE_WS_RMSNORM);
    if (ws_bytes < L.dgp + sizeof(float) * kNormBlocks * d) return LMCE_EINVAL;
    dgp = reinterpret_cast<float*>(static_cast<char*>(ws) + L.dgp);
  }
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  return rmsnorm_bwd_impl(x, ldx, g, rinv, dh, lddh, N, d, dx, lddx, dg, accumulate_dg, dgp,
                          static_cast<cudaStream_t>(stream));
}

int lmhead_ce_fwd_rmsnorm(const lmce_bf16* x, int64_t ldx, const float* g, float eps, const lmce_bf16* W, int64_t N,
                          int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask, float softcap,
                          float* nll, float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (int rc = check_norm(x, ldx, g, N, d); rc) return rc;
  if (!ws || !aligned16(ws) || !(eps >= 0.0f) || !std::isfinite(eps)) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, LMCE_WS_RMSNORM | (row_mask ? LMCE_WS_MASKED : 0u));
  if (ws_bytes < L.total) return LMCE_EINVAL;
  char* w = static_cast<char*>(ws);
  lmce_bf16* hn = reinterpret_cast<lmce_bf16*>(w + L.hn);
  if (int rc = check_common(hn, d, W, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!nll) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = rmsnorm_fwd_impl(x, ldx, g, eps, N, d, hn, d, reinterpret_cast<float*>(w + L.rinv), s, di.sms); rc)
    return rc;
  return fwd_impl(hn, d, W, N, V, d, tgt, row_mask, softcap, nll, lse, ws, ws_bytes, stream, LMCE_WS_RMSNORM);
}

int lmhead_ce_fwd_bwd_rmsnorm(const lmce_bf16* x, int64_t ldx, const float* g, float eps, const lmce_bf16* W,
                              int64_t N, int64_t V, int64_t d, const int64_t* tgt, const uint8_t* row_mask,
                              float softcap, float grad_scale, float* nll, float* lse, lmce_bf16* dx, int64_t lddx,
                              float* dg, float* dW, int accumulate, void* ws, size_t ws_bytes, void* stream) {
  if (int rc = check_norm(x, ldx, g, N, d); rc) return rc;
  if (!ws || !aligned16(ws) || !(eps >= 0.0f) || !std::isfinite(eps)) return LMCE_EINVAL;
  if (dg && !dx) return LMCE_EINVAL;  // the gain's gradient comes with dx
  if (dx && (lddx < d || lddx % 8 != 0 || !aligned16(dx))) return LMCE_EINVAL;
  if (dg && (reinterpret_cast<uintptr_t>(dg) & 3u) != 0) return LMCE_EINVAL;
  if (dW && !aligned16(dW)) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, LMCE_WS_RMSNORM | (row_mask ? LMCE_WS_MASKED : 0u));
  if (ws_bytes < L.total) return LMCE_EINVAL;
  char* w = static_cast<char*>(ws);
  lmce_bf16* hn = reinterpret_cast<lmce_bf16*>(w + L.hn);
  lmce_bf16* dhn = reinterpret_cast<lmce_bf16*>(w + L.dhn);
  float* rinv = reinterpret_cast<float*>(w + L.rinv);
  if (int rc = check_common(hn, d, W, N, V, d, tgt, softcap, ws); rc) return rc;
  if (!nll || !lse || !std::isfinite(grad_scale)) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = rmsnorm_fwd_impl(x, ldx, g, eps, N, d, hn, d, rinv, s, di.sms); rc) return rc;
  if (int rc = fwd_bwd_impl(hn, d, W, N, V, d, tgt, row_mask, softcap, grad_scale, nll, lse, dx ? dhn : nullptr, dW,
                            accumulate, ws, ws_bytes, stream, LMCE_WS_RMSNORM);
      rc)
    return rc;
  if (!dx) return LMCE_OK;
  return rmsnorm_bwd_impl(x, ldx, g, rinv, dhn, d, N, d, dx, lddx, dg, accumulate,
                          reinterpret_cast<float*>(w + L.dgp), s);
}

// The bpb reduction's arrival counter: bytes 8..11 of the workspace's 64-byte
// header (after the status word), zero from the caller's zero-fill and
// reset by every reduction.
unsigned* bpb_counter(void* ws) { return reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 8); }

int bpb_reduce(const float* nll, const int32_t* bytes, const uint8_t* row_mask, int64_t N, lmce_bpb_acc* acc,
               void* ws, size_t ws_bytes, void* stream) {
  if (!nll || !bytes || !acc || !ws || N < 1) return LMCE_EINVAL;
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(acc) & 7u) != 0) return LMCE_EINVAL;
  const Layout L = make_layout(1, 1, 64, 0u);
  if (ws_bytes < L.bpb + sizeof(lmce::BpbPartial) * lmce::kBpbBlocks) return LMCE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* part = reinterpret_cast<lmce::BpbPartial*>(static_cast<char*>(ws) + L.bpb);
  lmce::count_launches(1);
  lmce::bpb_kernel<<<lmce::kBpbBlocks, lmce::kBpbThreads, 0, s>>>(
      nll, bytes, row_mask, N, part, reinterpret_cast<lmce::BpbPartial*>(acc), bpb_counter(ws));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bpb_reduce launch");
  return LMCE_OK;
}

int bpb_reduce_lut(const float* nll, const int64_t* tgt, const int32_t* lut, int64_t V, const uint8_t* row_mask,
                   int64_t N, lmce_bpb_acc* acc, void* ws, size_t ws_bytes, void* stream) {
  if (!nll || !tgt || !lut || !acc || !ws || N < 1 || V < 1) return LMCE_EINVAL;
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(acc) & 7u) != 0) return LMCE_EINVAL;
  const Layout L = make_layout(1, 1, 64, 0u);
  if (ws_bytes < L.bpb + sizeof(lmce::BpbPartial) * lmce::kBpbBlocks) return LMCE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  auto* part = reinterpret_cast<lmce::BpbPartial*>(w + L.bpb);
  lmce::count_launches(1);
  lmce::bpb_kernel<<<lmce::kBpbBlocks, lmce::kBpbThreads, 0, s>>>(
      nll, nullptr, row_mask, N, part, reinterpret_cast<lmce::BpbPartial*>(acc), bpb_counter(ws), tgt, lut, V,
      reinterpret_cast<unsigned*>(w + L.status));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bpb_reduce_lut launch");
  return LMCE_OK;
}

int lmce_wait_selftest(long long limit_cycles, int arrive, void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 64 || !aligned16(ws) || limit_cycles < 0) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  lmce::count_launches(1);
  lmce::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, arrive,
                                                                               static_cast<unsigned*>(ws));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait_selftest launch");
  return LMCE_OK;
}

int lmce_bpb(const lmce_bpb_acc* acc, double* bpb_out) {
  if (!acc || !bpb_out) return LMCE_EINVAL;
  if (acc->sum_bytes == 0) return LMCE_EDATA;
  *bpb_out = acc->sum_nll / (std::log(2.0) * static_cast<double>(acc->sum_bytes));
  return LMCE_OK;
}

int lmhead_int4_dequant(const uint8_t* Wq, const lmce_f16* scales, int64_t V, int64_t d, int group, lmce_bf16* out,
                        void* stream) {
  const lmce_qhead hd = int4_head(Wq, scales, group);
  return lmhead_qhead_dequant(&hd, V, d, out, stream);
}

int lmhead_tied_embed_bwd(const int64_t* ids, const lmce_bf16* g, int64_t ldg, int64_t N, int64_t V, int64_t d,
                          float* dW, void* ws, size_t ws_bytes, void* stream) {
  if (!ids || !g || !dW || !ws) return LMCE_EINVAL;
  if (N < 1 || V < 1 || d < 1) return LMCE_EINVAL;
  if (N > (int64_t(1) << 30) || V > (int64_t(1) << 30)) return LMCE_EINVAL;
  if (d % 64 != 0 || d > 512) return LMCE_ENOTSUP;
  if (ldg < d || ldg % 8 != 0) return LMCE_EINVAL;
  if (!aligned16(g) || !aligned16(dW) || !aligned16(ws)) return LMCE_EINVAL;
  const Layout L = make_layout(N, V, d, LMCE_WS_EMBED);
  if (ws_bytes < L.total) return LMCE_EINVAL;
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  namespace ek = lmce::embk;
  const ek::Layout E = ek::layout(N, V, d);
  char* w = static_cast<char*>(ws);
  char* e = w + L.embed;
  unsigned* status = reinterpret_cast<unsigned*>(w + L.status);
  int* hist = reinterpret_cast<int*>(e + E.hist);
  int* lrank = reinterpret_cast<int*>(e + E.lrank);
  int* offs = reinterpret_cast<int*>(e + E.offs);
  int* pbase = reinterpret_cast<int*>(e + E.pbase);
  int* gbase = reinterpret_cast<int*>(e + E.gbase);
  int* perm = reinterpret_cast<int*>(e + E.perm);
  float* part = reinterpret_cast<float*>(e + E.part);
  float* gpart = reinterpret_cast<float*>(e + E.gpart);
  int* pcnt = reinterpret_cast<int*>(e + E.pcnt);
  int* gcnt = reinterpret_cast<int*>(e + E.gcnt);
  int* powner = reinterpret_cast<int*>(e + E.powner);
  const int R = static_cast<int>(ek::chunk_rows(N)), C = static_cast<int>(ek::n_chunks(N));
  const int n = static_cast<int>(N), v = static_cast<int>(V), dd = static_cast<int>(d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int use_smem = V <= ek::kCountSmemV ? 1 : 0;
  const size_t count_smem = use_smem ? sizeof(int) * static_cast<size_t>(V) : 0;
  int* lb = reinterpret_cast<int*>(e + E.lb);
  const int nb = static_cast<int>(cdiv(V, 256));
  lmce::count_launches(4);
  if (R == 1024 && V <= ek::kWalkersMaxV)
    ek::count8_kernel<<<C, 256, sizeof(uint16_t) * ek::kWalkers * static_cast<size_t>(V), s>>>(
        ids, n, v, hist, lrank, status, lb, static_cast<int>(ek::lb_ints(V)));
  else
    ek::count_kernel<<<C, 256, count_smem, s>>>(ids, n, v, R, hist, lrank, status, use_smem, lb,
                                                static_cast<int>(ek::lb_ints(V)));
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess)
    err = launch_pdl(ek::tokscan_kernel, nb, 256, 0, s, hist, C, v, offs, pbase, gbase, gcnt, pcnt, powner, lb,
                     status);
  if (err == cudaSuccess)
    err = launch_pdl(ek::place_kernel, static_cast<int>(cdiv(N, 256)), 256, 0, s, ids, n, v, R,
                     static_cast<const int*>(hist), static_cast<const int*>(lrank), static_cast<const int*>(offs), perm);
  if (err == cudaSuccess)
    err = launch_pdl(ek::pieces_kernel, di.sms * 8, 256, 0, s, reinterpret_cast<const uint16_t*>(g),
                     static_cast<long long>(ldg), dd, v, static_cast<const int*>(offs), static_cast<const int*>(pbase),
                     static_cast<const int*>(gbase), static_cast<const int*>(powner), static_cast<const int*>(perm), part,
                     gpart, pcnt, gcnt, dW);
  if (err != cudaSuccess) return cuda_fail(err, "tied_embed launch");
  err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err, "tied_embed launch");
  return LMCE_OK;
}

int lmce_status(void* ws, void* stream, int* code) {
  if (!ws || !code) return LMCE_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  const unsigned zero = 0;
  e = cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status clear)");
  *code = (v & lmce::ST_ETIMEOUT) ? LMCE_ETIMEOUT : (v & lmce::ST_EDATA) ? LMCE_EDATA : LMCE_OK;
  return LMCE_OK;
}

const char* lmce_last_cuda_error(void) { return g_last_err.c_str(); }

unsigned long long lmce_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* lmce_strerror(int code) {
  switch (code) {
    case LMCE_OK: return "ok";
    case LMCE_EINVAL: return "invalid argument";
    case LMCE_ENOTSUP: return "unsupported shape, softcap or device";
    case LMCE_ECUDA: return "CUDA error";
    case LMCE_EDATA: return "invalid data (target out of range or no bytes)";
    case LMCE_ETIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---- forward without a caller workspace ------------------------------------
// For callers that cannot hand the library a device allocation: the scratch
// of the forward (status word, partial sums of e^s, target logits) lives in a
// file-scope device array instead.  Every GPU that loads this library holds
// the array until the process exits; all calls on a device share it.
namespace {

constexpr int64_t kNoAllocMaxRows = 65536;   // N limit of lmhead_ce_fwd_noalloc
constexpr int64_t kNoAllocMaxVocab = 8192;   // V limit
constexpr size_t kNoAllocPartOff = 256;      // [0, 256): status word
constexpr size_t kNoAllocPartBytes =
    sizeof(float) * 2 * ((kNoAllocMaxVocab + lmce::fwdk::BN - 1) / lmce::fwdk::BN) * kNoAllocMaxRows;
constexpr size_t kNoAllocStOff = kNoAllocPartOff + kNoAllocPartBytes;
constexpr size_t kNoAllocBytes = kNoAllocStOff + sizeof(float) * kNoAllocMaxRows;  // about 16.3 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the symbol's host-side name is not a device address).
int noalloc_scratch(int dev, unsigned char** out) {
  static std::mutex mu;
  static unsigned char* ptr[64] = {};
  if (dev < 0 || dev >= 64) return LMCE_ENOTSUP;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = ptr[dev];
  return LMCE_OK;
}

}  // namespace

extern "C" int lmhead_ce_fwd_noalloc(const lmce_bf16* h, int64_t ldh, const lmce_bf16* W, int64_t N, int64_t V,
                                     int64_t d, const int64_t* tgt, float softcap, float* nll, float* lse,
                                     void* stream) {
  if (!h || !W || !tgt || !nll) return LMCE_EINVAL;
  if (N < 1 || V < 1 || d < 1) return LMCE_EINVAL;
  if (N > kNoAllocMaxRows || V > kNoAllocMaxVocab) {
    g_last_err = "lmhead_ce_fwd_noalloc: N <= 65536 and V <= 8192 (size of its static scratch)";
    return LMCE_EINVAL;
  }
  if (d % 64 != 0 || d > 512) return LMCE_ENOTSUP;
  if (ldh < d || ldh % 8 != 0) return LMCE_EINVAL;
  if (!aligned16(h) || !aligned16(W)) return LMCE_EINVAL;
  if (!softcap_ok(softcap) || softcap_online(softcap, V)) return LMCE_ENOTSUP;  // fixed-shift form only
  DevInfo di;
  if (int rc = dev_info(&di); rc) return rc;
  unsigned char* scratch = nullptr;
  if (int rc = noalloc_scratch(di.dev, &scratch); rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* status = reinterpret_cast<unsigned*>(scratch);
  // The status word starts every call clear, so that the finalize below sees
  // only this call's expired waits (it writes NaN rows for them).
  cudaError_t e0 = cudaMemsetAsync(status, 0, sizeof(unsigned), s);
  if (e0 != cudaSuccess) return cuda_fail(e0, "lmhead_ce_fwd_noalloc status reset");

  CUtensorMap tm_h, tm_w;
  if (int rc = lmce::make_map_bf16_3d(&tm_h, h, d, N, ldh * 2, lmce::fwdk::BM, static_cast<uint32_t>(d / 64)); rc)
    return rc;
  if (int rc = lmce::make_map_bf16_3d(&tm_w, W, d, V, d * 2, lmce::fwdk::HALF_N, lmce::fwdk::SC); rc) return rc;
  lmce::fwdk::Params p{};
  p.N = static_cast<int>(N);
  p.n_rows = nullptr;
  p.V = static_cast<int>(V);
  p.d = static_cast<int>(d);
  p.KC = static_cast<int>(d / 64);
  p.VT = static_cast<int>(cdiv(V, lmce::fwdk::BN));
  p.N_pad = static_cast<int>(cdiv(N, lmce::fwdk::PAIR_ROWS) * lmce::fwdk::PAIR_ROWS);
  p.tgt = tgt;
  fwd_params_softcap(p, softcap);
  p.part = reinterpret_cast<float*>(scratch + kNoAllocPartOff);
  p.partm = nullptr;
  p.st = reinterpret_cast<float*>(scratch + kNoAllocStOff);
  p.status = status;
  p.maxseg = p.VT;
  const int64_t T_max = cdiv(N, lmce::fwdk::PAIR_ROWS) * p.VT;
  const int pairs = static_cast<int>(std::min<int64_t>(T_max, lmce::fwdk::max_clusters(di.dev, di.sms)));
  lmce::count_launches(2);
  if (int rc = lmce::fwdk::launch(tm_h, tm_w, p, pairs, s); rc) return rc;
  const int fblocks = static_cast<int>(std::min<int64_t>(cdiv(N, 256), int64_t(di.sms) * 4));
  lmce::fwd_finalize_kernel<<<fblocks, 256, 0, s>>>(p.part, p.VT, pairs, lmce::fwdk::PAIR_ROWS, p.N_pad, p.st, tgt,
                                                    nullptr, static_cast<int>(N), static_cast<int>(V), nullptr, nll,
                                                    lse, status, /*nan_on_timeout=*/1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lmhead_ce_fwd_noalloc launch");
  return LMCE_OK;
}
