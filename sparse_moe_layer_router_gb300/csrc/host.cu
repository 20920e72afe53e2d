// host.cu -- the C ABI of libmoe_gb300 (declared in include/moe.h).
//
// Validates shapes and pointers on the host (nothing is launched on an
// error), lays out the caller's workspace, encodes TMA tensor maps and
// launches the kernels on the caller's stream.  The library allocates no
// device memory and keeps no state besides per-device constants.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"

namespace {

using namespace moe;

// Workspace header: status word (int32 at 0); router counters (int32 at 4:
// tokens re-decided at level 2, at 8: tokens that needed level 3).
constexpr size_t kHeader = 256;
// Router logits: split K until about this many CTAs run (half the SMs: fewer
// split partials for the select kernel to add; measured best of 76..608).
constexpr int kRouterTargetCtas = 76;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- devices
struct DevInfo {
  int checked = 0;
  int ok = 0;
  int sms = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

int current_device(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    d.sms = sms;
    d.checked = 1;
  }
  if (!d.ok) return MOE_ERR_UNSUPPORTED;
  *out = d;
  return MOE_OK;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Row-major bf16 matrix [rows][cols] as a 2-D map with a {64, box_rows} box, 128-B swizzle.
bool map_2d_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Gate/up weights [groups][2*half][cols] bf16 as a 4-D map {64-element K
// chunk, 16 rows, gate/up, 16-row block}: one {64, 16, 2, 4} box is a whole
// 64-feature k-block stage (four blocks of 16 gate rows followed by their 16
// up rows, 16 KB), one copy where the 3-D map takes four.
bool map_gate_up_bf16_4d(CUtensorMap* m, const void* base, uint64_t groups, uint64_t half,
                         uint64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const uint64_t rb = cols * 2;  // bytes per row
  const cuuint64_t dims[4] = {cols, 16, 2, groups * 2 * half / 16};
  const cuuint64_t strides[3] = {rb, half * rb, 16 * rb};
  const cuuint32_t box[4] = {64, 16, 2, 4};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed int4 weights [rows][cols/8] int32: 2-D map with a {32 words = 256
// values = 128 B, box_rows} box and the 128-byte swizzle.
bool map_2d_i4(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols / 8, rows};
  const cuuint64_t strides[1] = {cols / 2};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed int4 gate/up weights [groups][2*half][cols/8] as a 3-D map {cols/8
// words, groups*2*half rows, 2} whose third axis steps from a gate row to the
// matching up row (half rows further): a {32 words, 16, 2} box is 16 gate rows
// followed by the 16 matching up rows (128-byte swizzle).
bool map_gate_up_i4(CUtensorMap* m, const void* base, uint64_t groups, uint64_t half,
                    uint64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cols / 8, groups * 2 * half, 2};
  const cuuint64_t strides[2] = {cols / 2, half * (cols / 2)};
  const cuuint32_t box[3] = {32, 16, 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 group scales [rows][ngrp]: 2-D map with a {ngrp, box_rows} box (whole
// rows of scales), or the 3-D gate/up pairing with a {ngrp, 16, 2} box.
bool map_scales(CUtensorMap* m, const void* base, uint64_t groups, uint64_t rows_per_group,
                uint64_t ngrp, bool gate_up) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  if (gate_up) {
    const uint64_t half = rows_per_group / 2;
    const cuuint64_t dims[3] = {ngrp, groups * rows_per_group, 2};
    const cuuint64_t strides[2] = {ngrp * 2, half * ngrp * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(ngrp), 16, 2};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
  }
  const cuuint64_t dims[2] = {ngrp, groups * rows_per_group};
  const cuuint64_t strides[1] = {ngrp * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(ngrp), 128};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- validation
int validate(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->D < 1 || c->E < 1 || c->I < 1 || c->I_shared < 1 || c->k < 1 || c->k > c->E)
    return MOE_ERR_INVALID_ARG;
  if (c->T > (1 << 20) || c->E > 1024 || c->k > 32) return MOE_ERR_UNSUPPORTED;
  if (c->D % 128 != 0 || c->D > 65536) return MOE_ERR_UNSUPPORTED;
  if (c->I > 65536 || c->I_shared > 65536) return MOE_ERR_UNSUPPORTED;
  if (c->quant == MOE_QUANT_BF16) {
    if (c->I % 64 != 0 || c->I_shared % 64 != 0) return MOE_ERR_UNSUPPORTED;
  } else if (c->quant == MOE_QUANT_W4A16) {
    // symmetric int4 with group-128 scales along K or channel-wise scales
    // (group 0, one per output row); other layouts are rejected, as
    // unsupported quantisation formats are rejected at model load.  K tiles of
    // 256 packed values: D, I and I_shared multiples of 256
    if ((c->group != 128 && c->group != 0) || c->D % 256 != 0 || c->I % 256 != 0 ||
        c->I_shared % 256 != 0)
      return MOE_ERR_UNSUPPORTED;
  } else {
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// ---------------------------------------------------------------- workspace
// Router logits on the tensor cores: CTAs of 128 experts x 64 tokens, split
// over K (k-blocks of 64) until about kRouterTargetCtas CTAs run.
struct RouterPlan {
  int S = 1;
  int kb_per_split = 1;
};

RouterPlan router_plan(const moe_config* c) {
  RouterPlan r;
  const int nkb = c->D / 64;
  const long base = static_cast<long>((c->E + 127) / 128) * ((c->T + 63) / 64);
  long S = (kRouterTargetCtas + base - 1) / base;
  if (S > 16) S = 16;
  if (S > nkb) S = nkb;
  if (S < 1) S = 1;
  r.kb_per_split = (nkb + static_cast<int>(S) - 1) / static_cast<int>(S);
  r.S = (nkb + r.kb_per_split - 1) / r.kb_per_split;
  return r;
}

struct Layout {
  size_t blob = 0, zpart = 0, xnorm = 0, wnorm = 0;            // route
  size_t chunk = 0;                                              // permute
  size_t counts = 0, offsets = 0, perm = 0, inv = 0;             // forward
  size_t xperm = 0, h = 0, hs = 0, o = 0, os = 0, xin = 0, yout = 0;
  size_t total = 0;
};

struct Carver {
  size_t cur = kHeader;
  size_t take(size_t bytes) {
    const size_t at = cur;
    cur = align_up(cur + bytes, 256);
    return at;
  }
};

Layout layout(const moe_config* c, int entry) {
  Layout L;
  Carver cv;
  const size_t T = c->T, D = c->D, E = c->E, k = c->k, P = T * k;
  const size_t I = c->I, Is = c->I_shared;
  const RouterPlan rp = router_plan(c);
  const size_t chunks = (P + kPermuteChunk - 1) / kPermuteChunk;
  auto route_part = [&] {
    L.zpart = cv.take(static_cast<size_t>(rp.S) * T * E * 4);
    L.xnorm = cv.take(T * 4);  // sums of squares of the token rows
    L.wnorm = cv.take(E * 4);  // and of the router rows
  };
  switch (entry) {
    case MOE_ENTRY_ROUTE:
      route_part();
      break;
    case MOE_ENTRY_PERMUTE:
      L.chunk = cv.take(chunks * E * 4);
      break;
    case MOE_ENTRY_GROUPED_GEMM:
      L.xperm = cv.take(P * D * 2);  // gathered activation rows when a_row_index is given
      L.offsets = cv.take((E + 1) * 4);  // the caller's offsets, clamped and monotone
      L.perm = cv.take(P * 4);           // the caller's perm_pair, clamped
      break;
    case MOE_ENTRY_FORWARD_EXPERTS:
      L.chunk = cv.take(chunks * E * 4);
      L.counts = cv.take(E * 4);
      L.offsets = cv.take((E + 1) * 4);
      L.perm = cv.take(P * 4);
      L.inv = cv.take(P * 4);
      L.xperm = cv.take(P * D * 2);
      L.h = cv.take(P * I * 2);
      L.hs = cv.take(T * Is * 2);
      L.o = cv.take(P * D * 4);
      L.os = cv.take(T * D * 4);
      break;
    case MOE_ENTRY_FORWARD:
    case MOE_ENTRY_FORWARD_HOST:
      L.blob = cv.take(T * 2 * k * 4);
      route_part();
      L.chunk = cv.take(chunks * E * 4);
      L.counts = cv.take(E * 4);
      L.offsets = cv.take((E + 1) * 4);
      L.perm = cv.take(P * 4);
      L.inv = cv.take(P * 4);
      L.xperm = cv.take(P * D * 2);
      L.h = cv.take(P * I * 2);
      L.hs = cv.take(T * Is * 2);
      L.o = cv.take(P * D * 4);
      L.os = cv.take(T * D * 4);
      if (entry == MOE_ENTRY_FORWARD_HOST) {
        L.xin = cv.take(T * D * 2);
        L.yout = cv.take(T * D * 2);
      }
      break;
    default:
      return L;
  }
  L.total = cv.cur;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Error radius factor of the tensor-core router logits (see router.cu): at
// most 2^-15 of sum|x w| from each 64-wide chunk's accumulation, then every
// chunk value passes through at most h = kb_per_split + S + 2 fp32 roundings
// (running sum, split sum, bias); the fp64 index-order definition deviates from
// the exact sum by at most D * 2^-53 relative to sum |x_d w_d|.
float router_gamma(const moe_config* c, const RouterPlan& rp) {
  const double u = std::ldexp(1.0, -24);
  const double h = rp.kb_per_split + rp.S + 2.0;
  const double g = std::ldexp(1.0, -15) * (1.0 + std::ldexp(1.0, -10)) + h * u / (1.0 - h * u) +
                   c->D * std::ldexp(1.0, -53) * 1.01;
  return std::nextafter(static_cast<float>(g), INFINITY);
}

// Level-2 radius factor (router.cu, warp_dot_comp): the compensated sum's
// error-term chain has at most D/32 + 12 roundings over error terms totalling at
// most (D/32 + 33) u sum|x w|; add the fp64 index-order definition's own
// distance from the exact sum, (D + 2) 2^-53 sum|x w|.
float router_gamma2(const moe_config* c) {
  const double u = std::ldexp(1.0, -24);
  const double n1 = c->D / 32.0 + 12.0, n2 = c->D / 32.0 + 33.0;
  const double g = (n1 * u / (1.0 - n1 * u)) * n2 * u * 1.01 +
                   (c->D + 2.0) * std::ldexp(1.0, -53) * 1.01;
  return std::nextafter(static_cast<float>(g), INFINITY);
}

// Routes tokens [t0, t0 + n) of x into their rows of blob with the plan rp
// (split-K shape and radius).  Tokens are routed independently, so routing a
// batch in pieces with the whole batch's plan gives the bits of one call.
int route_rows(const moe_config* c, const RouterPlan& rp, const void* x, int t0, int n,
               const void* wr, const float* bias, int32_t* blob, void* ws, const Layout& L,
               cudaStream_t st) {
  const void* xr = static_cast<const char*>(x) + static_cast<size_t>(t0) * c->D * 2;
  int32_t* br = blob + static_cast<size_t>(t0) * 2 * c->k;
  float* zpart = at<float>(ws, L.zpart);
  float* xsq = at<float>(ws, L.xnorm);
  float* wsq = at<float>(ws, L.wnorm);
  CUtensorMap mw, mx;
  if (!map_2d_bf16(&mw, wr, c->E, c->D, 128) || !map_2d_bf16(&mx, xr, n, c->D, 64))
    return MOE_ERR_CUDA;
  const int rc = cuda_rc(launch_router_logits_tc(mw, mx, xr, wr, n, c->D, c->E, rp.S,
                                                 rp.kb_per_split, zpart, xsq, wsq,
                                                 at<int>(ws, 0), st));
  if (rc != MOE_OK) return rc;
  return cuda_rc(launch_router_select(zpart, rp.S, n, c->D, c->E, c->k, bias, xsq, wsq,
                                      router_gamma(c, rp), router_gamma2(c), xr, wr, br,
                                      at<int>(ws, 4), st));
}

// Clears the two refinement counters for this call.  The status word before
// them is left alone: an error recorded by an earlier call stays until
// moe_get_status reads it.
int clear_route_counters(void* ws, cudaStream_t st) {
  return cudaMemsetAsync(static_cast<char*>(ws) + 4, 0, 8, st) == cudaSuccess ? MOE_OK
                                                                               : MOE_ERR_CUDA;
}

int route_impl(const moe_config* c, const DevInfo&, const void* x, const void* wr,
               const float* bias, int32_t* blob, void* ws, const Layout& L, cudaStream_t st) {
  const int rc = clear_route_counters(ws, st);
  if (rc) return rc;
  return route_rows(c, router_plan(c), x, 0, c->T, wr, bias, blob, ws, L, st);
}

int choose_bn_max(const moe_config* c) {
  const double avg = static_cast<double>(c->T) * c->k / c->E;
  return (c->T >= 2048 || avg >= 48.0) ? 256 : 64;
}

// The second stream of split bf16 launches, with the events that fork it from
// and join it back to the caller's stream: one set per host thread and
// context, created on first use (in relaxed capture mode, so that a first use
// inside a stream capture is legal) and kept for the process.
struct SideStream {
  unsigned long long ctx;
  cudaStream_t stream;
  cudaEvent_t fork, join;
};
thread_local std::vector<SideStream> t_side_streams;

// Destroys this thread's set for the current context (moe_release_cache).
int release_side_streams() {
  unsigned long long id = 0;
  if (current_context_id(&id) != cudaSuccess) return MOE_ERR_CUDA;
  int rc = MOE_OK;
  for (size_t i = 0; i < t_side_streams.size();) {
    const SideStream& x = t_side_streams[i];
    if (x.ctx != id) {
      ++i;
      continue;
    }
    if (cudaEventDestroy(x.fork) != cudaSuccess || cudaEventDestroy(x.join) != cudaSuccess ||
        cudaStreamDestroy(x.stream) != cudaSuccess)
      rc = MOE_ERR_CUDA;
    t_side_streams.erase(t_side_streams.begin() + static_cast<long>(i));
  }
  return rc;
}

int side_stream(SideStream* out) {
  unsigned long long id = 0;
  if (current_context_id(&id) != cudaSuccess) return MOE_ERR_CUDA;
  for (const SideStream& x : t_side_streams)
    if (x.ctx == id) {
      *out = x;
      return MOE_OK;
    }
  SideStream x{id, nullptr, nullptr, nullptr};
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return MOE_ERR_CUDA;
  const bool ok = cudaStreamCreateWithFlags(&x.stream, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) == cudaSuccess;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess || !ok) return MOE_ERR_CUDA;
  t_side_streams.push_back(x);
  *out = x;
  return MOE_OK;
}

// Whether a launch takes the split below: bf16 with 256-row tiles and few
// enough rows per expert on average (under 8 * kSplitRows) that groups below
// kSplitRows rows are likely.  When every group is hot the split only adds its
// plan kernel and the fork and join (about 10 us per launch, measured at
// T = 8192 on 512 experts), so the dense shapes keep the single launch.
bool use_split(const moe_config* c, int bn_max) {
  return c->quant == MOE_QUANT_BF16 && bn_max == 256 &&
         static_cast<long>(c->T) * c->k < 8L * kSplitRows * c->E;
}

// A bf16 launch with 256-row tiles as two concurrent grids: groups of at least
// kSplitRows rows (tensor-bound) on the caller's stream, the smaller ones
// (weight-stream-bound, 64-row tiles and the deeper ring) on the side stream;
// the kernels share the SMs between them on the device.
// gh: a device int for the plan (bytes 12..15 of the workspace header).
int launch_split(GemmParams p, const GemmMaps& maps, const DevInfo& dev, int* gh,
                 cudaStream_t st) {
  SideStream ss;
  int rc = side_stream(&ss);
  if (rc) return rc;
  p.split_gh = gh;
  rc = cuda_rc(launch_split_plan(p, dev.sms, gh, st));
  if (rc) return rc;
  if (cudaEventRecord(ss.fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(ss.stream, ss.fork, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  p.split_role = 1;
  rc = cuda_rc(launch_grouped_gemm(p, maps, 256, MOE_QUANT_BF16, dev.sms, st));
  if (rc) return rc;
  p.split_role = 2;
  rc = cuda_rc(launch_grouped_gemm(p, maps, 64, MOE_QUANT_BF16, dev.sms, ss.stream));
  if (rc) return rc;
  if (cudaEventRecord(ss.join, ss.stream) != cudaSuccess ||
      cudaStreamWaitEvent(st, ss.join, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// One grouped GEMM launch over `n_groups` routed groups (a->offsets holds
// n_groups + 1 row offsets; a->w holds n_groups experts) plus, when
// a->a_shared is set, a shared group of `t_shared` rows.
int gemm_impl(const moe_config* c, const DevInfo& dev, const moe_gemm_args* a, void* ws,
              const Layout& L, cudaStream_t st, void* xperm_override, int n_groups,
              int t_shared) {
  const int P = c->T * c->k;
  const bool gate_up = a->op == MOE_OP_GATE_UP_SWIGLU;
  const bool has_shared = a->a_shared != nullptr;
  const bool w4 = c->quant == MOE_QUANT_W4A16;
  const void* b_routed = a->a;
  if (a->a_row_index) {
    if (!gate_up) return MOE_ERR_INVALID_ARG;
    void* xp = xperm_override ? xperm_override : at<void>(ws, L.xperm);
    const int grc = cuda_rc(launch_gather_rows(a->a, a->a_row_index, P, c->D, 1, c->T, xp,
                                               nullptr, nullptr, at<int>(ws, 0), st));
    if (grc) return grc;
    b_routed = xp;
  }
  GemmMaps maps;
  GemmParams p{};
  p.op = gate_up ? kOpGateUp : kOpDown;
  p.E = n_groups;
  p.has_shared = has_shared ? 1 : 0;
  p.T_shared = t_shared;
  p.offsets = a->offsets;
  p.perm_pair = a->perm_pair;
  p.blob = a->blob;
  p.k = c->k;
  p.status = at<int>(ws, 0);
  p.out = a->out;
  p.out_s = a->out_shared;
  p.wscale = static_cast<const uint16_t*>(a->w_scales);
  p.wscale_s = static_cast<const uint16_t*>(a->ws_scales);
  p.K = gate_up ? c->D : c->I;
  p.K_s = gate_up ? c->D : c->I_shared;
  // channel-wise scales: the restore leaves q unscaled and the epilogue
  // multiplies each accumulator row by its row's scale
  p.channel = (w4 && c->group == 0) ? 1 : 0;
  p.group = (w4 && c->group > 0) ? c->group : 128;
  const int bn_max = choose_bn_max(c);
  // The W4A16 64-row kernel copies token rows in 32-row boxes; the others
  // copy a tile's rows in power-of-two boxes of 16 to 128 rows (maps b..b8).
  const uint32_t tok_rows = (w4 && bn_max == 64) ? 32 : 16;
  const bool p2_boxes = !w4 || bn_max == 256;
  bool ok = true;
  if (gate_up) {
    p.m_tiles = c->I / 64;
    p.m_tiles_s = c->I_shared / 64;
    p.k_blocks = p.k_blocks_s = c->D / 64;
    p.a_rows_per_expert = 2 * c->I;
    p.ld_out = c->I;
    p.ld_out_s = c->I_shared;
    ok &= w4 ? map_gate_up_i4(&maps.a, a->w, n_groups, c->I, c->D)
             : map_gate_up_bf16_4d(&maps.a, a->w, n_groups, c->I, c->D);
    ok &= map_2d_bf16(&maps.b, b_routed, P, c->D, tok_rows);
    if (p2_boxes) {
      ok &= map_2d_bf16(&maps.b2, b_routed, P, c->D, 32);
      ok &= map_2d_bf16(&maps.b4, b_routed, P, c->D, 64);
      ok &= map_2d_bf16(&maps.b8, b_routed, P, c->D, 128);
    }
    if (has_shared) {
      ok &= w4 ? map_gate_up_i4(&maps.a_s, a->w_shared, 1, c->I_shared, c->D)
               : map_gate_up_bf16_4d(&maps.a_s, a->w_shared, 1, c->I_shared, c->D);
      ok &= map_2d_bf16(&maps.b_s, a->a_shared, t_shared, c->D, tok_rows);
      if (p2_boxes) {
        ok &= map_2d_bf16(&maps.b2_s, a->a_shared, t_shared, c->D, 32);
        ok &= map_2d_bf16(&maps.b4_s, a->a_shared, t_shared, c->D, 64);
        ok &= map_2d_bf16(&maps.b8_s, a->a_shared, t_shared, c->D, 128);
      }
    }
  } else {
    p.m_tiles = c->D / 128;
    p.m_tiles_s = c->D / 128;
    p.k_blocks = c->I / 64;
    p.k_blocks_s = c->I_shared / 64;
    p.a_rows_per_expert = c->D;
    p.ld_out = c->D;
    p.ld_out_s = c->D;
    ok &= w4 ? map_2d_i4(&maps.a, a->w, static_cast<uint64_t>(n_groups) * c->D, c->I, 128)
             : map_2d_bf16(&maps.a, a->w, static_cast<uint64_t>(n_groups) * c->D, c->I, 128);
    ok &= map_2d_bf16(&maps.b, b_routed, P, c->I, tok_rows);
    if (p2_boxes) {
      ok &= map_2d_bf16(&maps.b2, b_routed, P, c->I, 32);
      ok &= map_2d_bf16(&maps.b4, b_routed, P, c->I, 64);
      ok &= map_2d_bf16(&maps.b8, b_routed, P, c->I, 128);
    }
    if (has_shared) {
      ok &= w4 ? map_2d_i4(&maps.a_s, a->w_shared, c->D, c->I_shared, 128)
               : map_2d_bf16(&maps.a_s, a->w_shared, c->D, c->I_shared, 128);
      ok &= map_2d_bf16(&maps.b_s, a->a_shared, t_shared, c->I_shared, tok_rows);
      if (p2_boxes) {
        ok &= map_2d_bf16(&maps.b2_s, a->a_shared, t_shared, c->I_shared, 32);
        ok &= map_2d_bf16(&maps.b4_s, a->a_shared, t_shared, c->I_shared, 64);
        ok &= map_2d_bf16(&maps.b8_s, a->a_shared, t_shared, c->I_shared, 128);
      }
    }
  }
  // W4A16 scale tables by TMA when every K of the launch is a multiple of 1024
  // up to 4096 (whole rows of 8..32 scales, 16..64 B) and the 64-row variant runs.
  const bool k_ok = p.K % 1024 == 0 && p.K <= 4096 && (!has_shared || (p.K_s % 1024 == 0 &&
                                                                      p.K_s <= 4096));
  p.scale_table = (w4 && !p.channel && bn_max == 64 && k_ok) ? 1 : 0;
  if (p.scale_table) {
    const uint64_t rows_r = gate_up ? 2ull * c->I : static_cast<uint64_t>(c->D);
    ok &= map_scales(&maps.sc, a->w_scales, n_groups, rows_r, p.K / c->group, gate_up);
    if (has_shared) {
      const uint64_t rows_s = gate_up ? 2ull * c->I_shared : static_cast<uint64_t>(c->D);
      ok &= map_scales(&maps.sc_s, a->ws_scales, 1, rows_s, p.K_s / c->group, gate_up);
    }
  }
  if (!ok) return MOE_ERR_CUDA;
  if (!p2_boxes) maps.b2 = maps.b4 = maps.b8 = maps.b;
  if (!has_shared) {
    maps.a_s = maps.a;
    maps.b_s = maps.b;
  }
  if (!p2_boxes || !has_shared) maps.b2_s = maps.b4_s = maps.b8_s = maps.b_s;
  if (!p.scale_table || !has_shared) maps.sc_s = maps.a_s;
  if (!p.scale_table) maps.sc = maps.a;
  if (use_split(c, bn_max)) return launch_split(p, maps, dev, at<int>(ws, 12), st);
  return cuda_rc(launch_grouped_gemm(p, maps, bn_max, c->quant, dev.sms, st));
}

int check_gemm_args(const moe_config* c, const moe_gemm_args* a) {
  if (!a || !a->a || !a->offsets || !a->w || !a->out) return MOE_ERR_INVALID_ARG;
  if (a->op != MOE_OP_GATE_UP_SWIGLU && a->op != MOE_OP_DOWN_WEIGHTED) return MOE_ERR_INVALID_ARG;
  if (a->op == MOE_OP_DOWN_WEIGHTED && (!a->perm_pair || !a->blob)) return MOE_ERR_INVALID_ARG;
  if (a->a_shared && (!a->w_shared || !a->out_shared)) return MOE_ERR_INVALID_ARG;
  if (c->quant == MOE_QUANT_W4A16 && (!a->w_scales || (a->a_shared && !a->ws_scales)))
    return MOE_ERR_INVALID_ARG;
  if (c->quant == MOE_QUANT_BF16 && (a->w_scales || a->ws_scales)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {a->a, a->w, a->w_scales, a->out, a->a_shared, a->w_shared, a->ws_scales,
                        a->out_shared, a->offsets};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

int check_weights(const moe_config* c, const moe_weights* w) {
  if (!w || !w->w_router || !w->w_gate_up || !w->w_down || !w->ws_gate_up || !w->ws_down)
    return MOE_ERR_INVALID_ARG;
  if (c->quant == MOE_QUANT_W4A16 &&
      (!w->s_gate_up || !w->s_down || !w->ss_gate_up || !w->ss_down))
    return MOE_ERR_INVALID_ARG;
  if (c->quant == MOE_QUANT_BF16 && (w->s_gate_up || w->s_down || w->ss_gate_up || w->ss_down))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {w->w_router, w->w_gate_up, w->w_down, w->s_gate_up, w->s_down,
                        w->ws_gate_up, w->ws_down, w->ss_gate_up, w->ss_down};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

// The whole layer on `st`; with route = false the blob in ws is already
// written, and with combine = false it stops after the down GEMM (o and
// o_shared in ws) and y is not written.
int forward_impl(const moe_config* c, const DevInfo& dev, const void* x, const moe_weights* w,
                 void* y, void* ws, const Layout& L, cudaStream_t st, bool combine = true,
                 bool route = true) {
  int rc = MOE_OK;
  if (route) {
    rc = route_impl(c, dev, x, w->w_router, w->router_bias, at<int32_t>(ws, L.blob), ws, L, st);
    if (rc) return rc;
  }
  rc = cuda_rc(launch_permute(at<int32_t>(ws, L.blob), c->T, c->k, c->E, at<int32_t>(ws, L.chunk),
                              at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                              at<int32_t>(ws, L.perm), at<int32_t>(ws, L.inv), at<int>(ws, 0), st));
  if (rc) return rc;
  // dispatch: token rows in grouped order (scatter from T = 2048: skewed step
  // -1.2%; the row gather below it: decode 5 us faster than the scatter)
  rc = cuda_rc(launch_dispatch_rows(x, at<int32_t>(ws, L.perm), at<int32_t>(ws, L.inv), c->T,
                                    c->k, c->D, at<void>(ws, L.xperm), nullptr, nullptr, nullptr,
                                    st));
  if (rc) return rc;
  moe_gemm_args g{};
  g.op = MOE_OP_GATE_UP_SWIGLU;
  g.a = at<void>(ws, L.xperm);
  g.offsets = at<int32_t>(ws, L.offsets);
  g.w = w->w_gate_up;
  g.w_scales = w->s_gate_up;
  g.out = at<void>(ws, L.h);
  g.a_shared = x;
  g.w_shared = w->ws_gate_up;
  g.ws_scales = w->ss_gate_up;
  g.out_shared = at<void>(ws, L.hs);
  rc = gemm_impl(c, dev, &g, ws, L, st, nullptr, c->E, c->T);
  if (rc) return rc;
  moe_gemm_args d{};
  d.op = MOE_OP_DOWN_WEIGHTED;
  d.a = at<void>(ws, L.h);
  d.offsets = at<int32_t>(ws, L.offsets);
  d.w = w->w_down;
  d.w_scales = w->s_down;
  d.perm_pair = at<int32_t>(ws, L.perm);
  d.blob = at<int32_t>(ws, L.blob);
  d.out = at<void>(ws, L.o);
  d.a_shared = at<void>(ws, L.hs);
  d.w_shared = w->ws_down;
  d.ws_scales = w->ss_down;
  d.out_shared = at<void>(ws, L.os);
  rc = gemm_impl(c, dev, &d, ws, L, st, nullptr, c->E, c->T);
  if (rc || !combine) return rc;
  return cuda_rc(launch_combine(at<float>(ws, L.o), at<float>(ws, L.os), at<int32_t>(ws, L.inv),
                                c->T, c->T * c->k, c->D, c->k, y, st));
}

// moe_forward_host's first step: x copied into the workspace and routed.  From
// T = 4096 the copy runs in chunks of 2048 tokens on the library's second
// stream, and each chunk is routed on `st` once it has arrived (with the whole
// batch's router plan), overlapping the copy of the chunks after it.  The copy
// is bound by the host link; a route call costs more per token on fewer
// tokens (53 us for 1024, 165 us for 8192), and 2048-token chunks keep that
// extra cost below what the overlap saves.
int host_copy_and_route(const moe_config* c, const void* x_host, void* xd, const moe_weights* w,
                        void* ws, const Layout& L, cudaStream_t st) {
  const size_t row = static_cast<size_t>(c->D) * 2;
  const RouterPlan rp = router_plan(c);
  int32_t* blob = at<int32_t>(ws, L.blob);
  int rc = clear_route_counters(ws, st);
  if (rc) return rc;
  constexpr int kChunk = 2048;
  if (c->T < 2 * kChunk) {
    if (cudaMemcpyAsync(xd, x_host, c->T * row, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    return route_rows(c, rp, xd, 0, c->T, w->w_router, w->router_bias, blob, ws, L, st);
  }
  SideStream ss;
  rc = side_stream(&ss);
  if (rc) return rc;
  // the copies start after the work already queued on `st` (it may still read ws)
  if (cudaEventRecord(ss.fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(ss.stream, ss.fork, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  for (int t0 = 0; t0 < c->T; t0 += kChunk) {
    const int n = std::min(kChunk, c->T - t0);
    if (cudaMemcpyAsync(static_cast<char*>(xd) + t0 * row,
                        static_cast<const char*>(x_host) + t0 * row, n * row,
                        cudaMemcpyHostToDevice, ss.stream) != cudaSuccess ||
        cudaEventRecord(ss.join, ss.stream) != cudaSuccess ||
        cudaStreamWaitEvent(st, ss.join, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    rc = route_rows(c, rp, xd, t0, n, w->w_router, w->router_bias, blob, ws, L, st);
    if (rc) return rc;
  }
  return MOE_OK;
}

// moe_forward_host's last step: the combine in chunks of tokens, each chunk's
// copy to the host queued on the library's second stream as soon as the
// chunk is combined, so that the copies (bound by the host link) overlap the
// combine of the chunks after them.  Chunks of at least 256 tokens, at most 8.
int combine_to_host(const moe_config* c, void* ws, const Layout& L, void* y_dev, void* y_host,
                    cudaStream_t st) {
  const int P = c->T * c->k;
  const size_t row = static_cast<size_t>(c->D) * 2;
  const int nc = std::max(1, std::min(8, c->T / 256));
  if (nc == 1) {
    const int rc = cuda_rc(launch_combine(at<float>(ws, L.o), at<float>(ws, L.os),
                                          at<int32_t>(ws, L.inv), c->T, P, c->D, c->k, y_dev, st));
    if (rc) return rc;
    return cudaMemcpyAsync(y_host, y_dev, c->T * row, cudaMemcpyDeviceToHost, st) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  SideStream ss;
  int rc = side_stream(&ss);
  if (rc) return rc;
  const int tc = (c->T + nc - 1) / nc;
  for (int t0 = 0; t0 < c->T; t0 += tc) {
    const int n = std::min(tc, c->T - t0);
    rc = cuda_rc(launch_combine(at<float>(ws, L.o), at<float>(ws, L.os) + static_cast<size_t>(t0) * c->D,
                                at<int32_t>(ws, L.inv) + static_cast<size_t>(t0) * c->k, n, P, c->D,
                                c->k, static_cast<char*>(y_dev) + t0 * row, st));
    if (rc) return rc;
    if (cudaEventRecord(ss.fork, st) != cudaSuccess ||
        cudaStreamWaitEvent(ss.stream, ss.fork, 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(y_host) + t0 * row, static_cast<char*>(y_dev) + t0 * row,
                        n * row, cudaMemcpyDeviceToHost, ss.stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaEventRecord(ss.join, ss.stream) != cudaSuccess ||
      cudaStreamWaitEvent(st, ss.join, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Expert-parallel slice: dispatch every pair, but gather, compute and combine
// only the rows of experts [e0, e1) (local weights indexed e - e0) and the
// shared expert for tokens [s0, s1).
int forward_experts_impl(const moe_config* c, const DevInfo& dev, const void* x,
                         const int32_t* blob, const moe_weights* w, int e0, int e1, int s0, int s1,
                         float* y32, void* ws, const Layout& L, cudaStream_t st) {
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int rc = cuda_rc(launch_permute(blob, c->T, c->k, c->E, at<int32_t>(ws, L.chunk),
                                  at<int32_t>(ws, L.counts), offsets, at<int32_t>(ws, L.perm),
                                  at<int32_t>(ws, L.inv), at<int>(ws, 0), st));
  if (rc) return rc;
  // grouped rows of the local experts: [offsets[e0], offsets[e1])
  const int32_t* row_lo = offsets + e0;
  const int32_t* row_hi = offsets + e1;
  rc = cuda_rc(launch_dispatch_rows(x, at<int32_t>(ws, L.perm), at<int32_t>(ws, L.inv), c->T,
                                    c->k, c->D, at<void>(ws, L.xperm), row_lo, row_hi, nullptr,
                                    st));
  if (rc) return rc;
  const int ts = s1 - s0;
  const void* x_sh = static_cast<const char*>(x) + static_cast<size_t>(s0) * c->D * 2;
  moe_gemm_args g{};
  g.op = MOE_OP_GATE_UP_SWIGLU;
  g.a = at<void>(ws, L.xperm);
  g.offsets = offsets + e0;
  g.w = w->w_gate_up;
  g.w_scales = w->s_gate_up;
  g.out = at<void>(ws, L.h);
  if (ts > 0) {
    g.a_shared = x_sh;
    g.w_shared = w->ws_gate_up;
    g.ws_scales = w->ss_gate_up;
    g.out_shared = at<void>(ws, L.hs);
  }
  rc = gemm_impl(c, dev, &g, ws, L, st, nullptr, e1 - e0, ts);
  if (rc) return rc;
  moe_gemm_args d{};
  d.op = MOE_OP_DOWN_WEIGHTED;
  d.a = at<void>(ws, L.h);
  d.offsets = offsets + e0;
  d.w = w->w_down;
  d.w_scales = w->s_down;
  d.perm_pair = at<int32_t>(ws, L.perm);
  d.blob = blob;
  d.out = at<void>(ws, L.o);
  if (ts > 0) {
    d.a_shared = at<void>(ws, L.hs);
    d.w_shared = w->ws_down;
    d.ws_scales = w->ss_down;
    d.out_shared = at<void>(ws, L.os);
  }
  rc = gemm_impl(c, dev, &d, ws, L, st, nullptr, e1 - e0, ts);
  if (rc) return rc;
  return cuda_rc(launch_combine_partial(at<float>(ws, L.o), ts > 0 ? at<float>(ws, L.os) : nullptr,
                                        at<int32_t>(ws, L.inv), c->T, c->D, c->k, row_lo, row_hi,
                                        s0, s1, y32, st));
}

int begin(const moe_config* c, int entry, void* ws, size_t ws_bytes, DevInfo* dev, Layout* L) {
  int rc = validate(c);
  if (rc) return rc;
  *L = layout(c, entry);
  if (!ws || ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  return current_device(dev);
}

}  // namespace

// Chained (programmatic dependent) launches for batches up to 32768 pairs.
static bool chain_launches(const moe_config* c) {
  return c && static_cast<long>(c->T) * c->k <= 32768;
}

extern "C" {

size_t moe_workspace_size(const moe_config* cfg, int entry) {
  if (validate(cfg) != MOE_OK) return 0;
  if (entry < MOE_ENTRY_ROUTE || entry > MOE_ENTRY_FORWARD_EXPERTS) return 0;
  return layout(cfg, entry).total;
}

int moe_route(const moe_config* cfg, const void* x, const void* w_router, const float* bias,
              int32_t* blob, void* ws, size_t ws_bytes, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  if (!x || !w_router || !blob) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(blob) || (bias && !aligned16(bias)))
    return MOE_ERR_ALIGN;
  DevInfo dev;
  Layout L;
  int rc = begin(cfg, MOE_ENTRY_ROUTE, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  return route_impl(cfg, dev, x, w_router, bias, blob, ws, L, static_cast<cudaStream_t>(stream));
}

int moe_router_logits(const moe_config* cfg, const void* x, const void* w_router, float* z,
                      void* ws, size_t ws_bytes, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  if (!x || !w_router || !z) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(z)) return MOE_ERR_ALIGN;
  DevInfo dev;
  Layout L;
  int rc = begin(cfg, MOE_ENTRY_ROUTE, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap mw, mx;
  if (!map_2d_bf16(&mw, w_router, cfg->E, cfg->D, 128) || !map_2d_bf16(&mx, x, cfg->T, cfg->D, 64))
    return MOE_ERR_CUDA;
  // one split: z itself is the split's output
  return cuda_rc(launch_router_logits_tc(mw, mx, x, w_router, cfg->T, cfg->D, cfg->E, 1,
                                         cfg->D / 64, z, at<float>(ws, L.xnorm),
                                         at<float>(ws, L.wnorm), at<int>(ws, 0), st));
}

int moe_permute(const moe_config* cfg, const int32_t* blob, int32_t* counts, int32_t* offsets,
                int32_t* perm_pair, int32_t* inv_row, const void* x, void* x_perm, void* ws,
                size_t ws_bytes, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  if (!blob || !counts || !offsets || !perm_pair || !inv_row) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_ALIGN;
  DevInfo dev;
  Layout L;
  int rc = begin(cfg, MOE_ENTRY_PERMUTE, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = cuda_rc(launch_permute(blob, cfg->T, cfg->k, cfg->E, at<int32_t>(ws, L.chunk), counts,
                              offsets, perm_pair, inv_row, at<int>(ws, 0), st));
  if (rc || !x) return rc;
  return cuda_rc(launch_dispatch_rows(x, perm_pair, inv_row, cfg->T, cfg->k, cfg->D, x_perm,
                                      nullptr, nullptr, nullptr, st));
}

int moe_permute_static(const moe_config* cfg, const int32_t* blob, int32_t* counts,
                       int32_t* offsets, int32_t* perm_pair, int32_t* inv_row, const void* x,
                       void* x_perm, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  if (!blob || !counts || !offsets || !perm_pair || !inv_row) return MOE_ERR_INVALID_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_ALIGN;
  const long P = static_cast<long>(cfg->T) * cfg->k;
  const long chunks = (P + kPermuteChunk - 1) / kPermuteChunk;
  if (chunks * cfg->E > kStaticPermuteScratchInts) return MOE_ERR_SCRATCH_LIMIT;
  DevInfo dev;
  rc = current_device(&dev);
  if (rc) return rc;
  return cuda_rc(launch_permute_static(blob, cfg->T, cfg->k, cfg->E, counts, offsets, perm_pair,
                                       inv_row, x, cfg->D, x_perm,
                                       static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm(const moe_config* cfg, const moe_gemm_args* args, void* ws, size_t ws_bytes,
                     void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  rc = check_gemm_args(cfg, args);
  if (rc) return rc;
  DevInfo dev;
  Layout L;
  rc = begin(cfg, MOE_ENTRY_GROUPED_GEMM, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  // The kernels trust offsets and perm_pair (the forward entries pass arrays
  // moe_permute wrote); caller arrays are first copied into range.
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe_gemm_args g = *args;
  g.offsets = at<int32_t>(ws, L.offsets);
  g.perm_pair = args->perm_pair ? at<int32_t>(ws, L.perm) : nullptr;
  rc = cuda_rc(launch_sanitize_gemm_indices(args->offsets, cfg->E + 1, cfg->T * cfg->k,
                                            at<int32_t>(ws, L.offsets), args->perm_pair,
                                            at<int32_t>(ws, L.perm), at<int>(ws, 0), st));
  if (rc) return rc;
  return gemm_impl(cfg, dev, &g, ws, L, st, nullptr, cfg->E, cfg->T);
}

int moe_combine(const moe_config* cfg, const float* o, const float* o_shared,
                const int32_t* inv_row, void* y, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  if (!o || !inv_row || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(y) || (o_shared && !aligned16(o_shared))) return MOE_ERR_ALIGN;
  DevInfo dev;
  rc = current_device(&dev);
  if (rc) return rc;
  return cuda_rc(launch_combine(o, o_shared, inv_row, cfg->T, cfg->T * cfg->k, cfg->D, cfg->k,
                                y, static_cast<cudaStream_t>(stream)));
}

int moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* y, void* ws,
                size_t ws_bytes, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_ALIGN;
  rc = check_weights(cfg, w);
  if (rc) return rc;
  DevInfo dev;
  Layout L;
  rc = begin(cfg, MOE_ENTRY_FORWARD, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  return forward_impl(cfg, dev, x, w, y, ws, L, static_cast<cudaStream_t>(stream));
}

int moe_forward_host(const moe_config* cfg, const void* x_host, const moe_weights* w, void* y_host,
                     void* ws, size_t ws_bytes, void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  rc = check_weights(cfg, w);
  if (rc) return rc;
  DevInfo dev;
  Layout L;
  rc = begin(cfg, MOE_ENTRY_FORWARD_HOST, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* xd = at<void>(ws, L.xin);
  void* yd = at<void>(ws, L.yout);
  rc = host_copy_and_route(cfg, x_host, xd, w, ws, L, st);
  if (rc) return rc;
  rc = forward_impl(cfg, dev, xd, w, yd, ws, L, st, false, false);
  if (rc) return rc;
  return combine_to_host(cfg, ws, L, yd, y_host, st);
}

int moe_forward_experts(const moe_config* cfg, const void* x, const int32_t* blob,
                        const moe_weights* w, int e_begin, int e_end, int shared_begin,
                        int shared_end, float* y_partial, void* ws, size_t ws_bytes,
                        void* stream) {
  PdlScope pdl_scope(chain_launches(cfg));
  int rc = validate(cfg);
  if (rc) return rc;
  if (!x || !blob || !w || !y_partial) return MOE_ERR_INVALID_ARG;
  if (e_begin < 0 || e_begin >= e_end || e_end > cfg->E) return MOE_ERR_INVALID_ARG;
  if (shared_begin < 0 || shared_begin > shared_end || shared_end > cfg->T)
    return MOE_ERR_INVALID_ARG;
  const bool sh = shared_end > shared_begin;
  if (!w->w_gate_up || !w->w_down || (sh && (!w->ws_gate_up || !w->ws_down)))
    return MOE_ERR_INVALID_ARG;
  const bool w4 = cfg->quant == MOE_QUANT_W4A16;
  if (w4 && (!w->s_gate_up || !w->s_down || (sh && (!w->ss_gate_up || !w->ss_down))))
    return MOE_ERR_INVALID_ARG;
  if (!w4 && (w->s_gate_up || w->s_down || w->ss_gate_up || w->ss_down))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, blob, y_partial, w->w_gate_up, w->w_down, w->s_gate_up, w->s_down,
                        w->ws_gate_up, w->ws_down, w->ss_gate_up, w->ss_down};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return MOE_ERR_ALIGN;
  DevInfo dev;
  Layout L;
  rc = begin(cfg, MOE_ENTRY_FORWARD_EXPERTS, ws, ws_bytes, &dev, &L);
  if (rc) return rc;
  return forward_experts_impl(cfg, dev, x, blob, w, e_begin, e_end, shared_begin, shared_end,
                              y_partial, ws, L, static_cast<cudaStream_t>(stream));
}

int moe_repack_int4(const int32_t* src, int32_t* dst, size_t n_words, int src_layout,
                    void* stream) {
  if (!src || !dst) return MOE_ERR_INVALID_ARG;
  if (src_layout != MOE_INT4_SEQUENTIAL && src_layout != MOE_INT4_SEQUENTIAL_OFFSET8)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGN;
  if (n_words == 0) return MOE_OK;
  DevInfo dev;
  const int rc = current_device(&dev);
  if (rc) return rc;
  return cuda_rc(launch_repack_int4(reinterpret_cast<const uint32_t*>(src),
                                    reinterpret_cast<uint32_t*>(dst), n_words,
                                    src_layout == MOE_INT4_SEQUENTIAL_OFFSET8,
                                    static_cast<cudaStream_t>(stream)));
}

int moe_get_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (h != 0 && cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
  return h;
}

int moe_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned int limit_ms, void* stream) {
  if (!ws || ws_bytes < kHeader) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_ALIGN;
  if (limit_ms < 1 || limit_ms > 10000) return MOE_ERR_INVALID_ARG;
  DevInfo dev;
  int rc = current_device(&dev);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_rc(launch_selftest_wait(at<int>(ws, 0), 1000000ull * limit_ms, st));
}

int moe_release_cache(void) { return release_side_streams(); }

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "success";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape, format or device";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_SCRATCH_LIMIT:
      return "problem larger than the fixed scratch of moe_permute_static";
    default: return "unknown error";
  }
}

}  // extern "C"
