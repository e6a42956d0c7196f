// specverify.cu -- C ABI of libspecverify (see include/specverify.h):
// argument checks, workspace layout, launch of the sm_103a kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "specverify.h"
#ifdef SV_NVTX
#include <nvtx3/nvToolsExt.h>
#endif
#include "sv_chain.cuh"
#include "sv_stats.cuh"
#include "sv_topk.cuh"
#include "sv_tree.cuh"
#include "sv_treemask.cuh"
#include "sv_treewalk.cuh"

namespace {

using namespace sv;

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct Layout {
  size_t tickets, jobs, partials, segsums, scratch, total;
};

static_assert(kDrawTicketBase == SV_MAX_B, "draw tickets follow the request tickets");
static_assert(static_cast<int64_t>(SV_MAX_V) / (kTkEpl * kTkMaxFold) * 4 <= kTkMapBytes,
              "the top-k map holds a row of SV_MAX_V fp32 logits in groups of 16 kTkMaxFold");
static_assert(sizeof(TopkShared) * kTkCtasPerSm + 2048 <= 228 * 1024,
              "the top-k pass keeps kTkCtasPerSm CTAs on an SM");
static_assert(2 * SV_MAX_K + 1 <= 96, "top-k finalize: row statistics in three lanes' strides");
static_assert(SV_MAX_V / kRSeg <= kMaxPages * kPageSeg && 2 * kMaxPages <= kMaxRowsPerReq,
              "draw finalize pages");

// The header, the tickets (requests, then their draws) and the draw records
// sit at fixed offsets with a fixed capacity
// (SV_MAX_B requests), so the region that every call leaves zeroed is the
// same for all problem sizes: one initialised workspace serves chain and
// tree calls of any shape, one call at a time.
Layout layout_for(int64_t partial_slots, int64_t segsum_floats, int64_t scratch_floats) {
  Layout L;
  L.tickets = align_up(sizeof(WsHeader));
  L.jobs = align_up(L.tickets + sizeof(unsigned int) * 2 * static_cast<size_t>(SV_MAX_B));
  L.partials = align_up(L.jobs + sizeof(unsigned long long) * kJobWords *
                                     static_cast<size_t>(SV_MAX_B));
  L.segsums = align_up(L.partials + sizeof(float2) * static_cast<size_t>(partial_slots));
  L.scratch = align_up(L.segsums + sizeof(float) * static_cast<size_t>(segsum_floats));
  L.total = align_up(L.scratch + sizeof(float) * static_cast<size_t>(scratch_floats));
  return L;
}

Ws ws_view(void* base, const Layout& L) {
  char* p = static_cast<char*>(base);
  Ws w;
  w.hdr = reinterpret_cast<WsHeader*>(p);
  w.tickets = reinterpret_cast<unsigned int*>(p + L.tickets);
  w.partials = reinterpret_cast<float2*>(p + L.partials);
  w.segsums = reinterpret_cast<float*>(p + L.segsums);
  w.jobs = reinterpret_cast<void*>(p + L.jobs);
  w.scratch = reinterpret_cast<float*>(p + L.scratch);
  return w;
}

int es_of(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }
int chunk_el_of(sv_dtype d) { return kChunkBytes / es_of(d); }
int resid_chunk_el_of(sv_dtype d) { return kChunkBytes / 2 / es_of(d); }

// Top-k pass: the length of a row's eight segments, and the scratch it
// writes (byte offsets within the scratch region): per row its list and
// (m, Z).
struct TopkLayout {
  int seg_len = 0;
  size_t lists = 0, mz = 0, bytes = 0;
};
TopkLayout topk_layout(int64_t B, int64_t K, int64_t V, int64_t max_top_k) {
  TopkLayout T;
  if (max_top_k <= 0) return T;
  const int64_t per = (V + kTkWarps - 1) / kTkWarps;
  T.seg_len = static_cast<int>((per + kTkSegAlign - 1) / kTkSegAlign * kTkSegAlign);
  const size_t rows = static_cast<size_t>(B) * (2 * K + 1);
  T.lists = 0;
  T.mz = align_up(T.lists + sizeof(float2) * rows * max_top_k);
  T.bytes = align_up(T.mz + sizeof(float2) * rows);
  return T;
}

// Chain calls: per-row chunk partials for the main pass, per-request
// segment sums for the draw pass, and the top-k pass's scratch.
Layout chain_layout(int64_t B, int64_t K, int64_t V, sv_dtype dtype, int64_t max_top_k) {
  const int64_t ipr = (V + chunk_el_of(dtype) - 1) / chunk_el_of(dtype);
  const int64_t ipr2 = (V + resid_chunk_el_of(dtype) - 1) / resid_chunk_el_of(dtype);
  return layout_for(B * (2 * K + 1) * ipr, B * ipr2 * (resid_chunk_el_of(dtype) / kRSeg),
                    static_cast<int64_t>(topk_layout(B, K, V, max_top_k).bytes / sizeof(float)));
}

Layout tree_layout(int64_t B, int64_t N, int64_t M, int64_t V, sv_dtype dtype) {
  const int64_t ipr = (V + chunk_el_of(dtype) - 1) / chunk_el_of(dtype);
  return layout_for(B * (N + M) * ipr, 0, B * 2 * V);
}

// Per-device facts, looked up once.
struct DeviceInfo {
  int sms = 0;
  bool supported = false;
};
std::mutex g_mu;
DeviceInfo g_dev[64];
bool g_known[64];

sv_status device_info(DeviceInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
  if (dev < 0 || dev >= 64) return SV_EUNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_known[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SV_ECUDA;
    g_dev[dev].sms = sms;
    g_dev[dev].supported = (major == 10 && minor == 3);
    g_known[dev] = true;
  }
  out = g_dev[dev];
  return out.supported ? SV_OK : SV_EUNSUPPORTED;
}

size_t pos_table_bytes(int n_req, int aux_bytes) {
  return (sizeof(float2) + aux_bytes) * n_req + sizeof(int) * n_req + sizeof(int) * (n_req + 1);
}

template <class P>
size_t kernel_smem(int n_req) {
  return 128 + static_cast<size_t>(kStages) * kChunkBytes +
         ((shared_bytes<P>() + 15) & ~size_t(15)) + pos_table_bytes(n_req, P::kAuxBytes);
}

template <class P>
sv_status launch(const P& prob, int grid, cudaStream_t stream) {
  const size_t smem = kernel_smem<P>(prob.n_req);
  if (cudaFuncSetAttribute(verify_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return SV_ECUDA;
  // Programmatic stream serialisation: the kernel waits for the preceding
  // work itself (griddepcontrol.wait), so its launch may overlap that work's
  // tail.  Cooperative: CTAs of this kernel wait on results other CTAs
  // publish (control CTAs on chunk partials, draw scouts on draw records),
  // so every CTA of the grid must be resident at once; a cooperative launch
  // guarantees that, or fails up front (SV_ECORESIDENT) when the grid
  // cannot fit -- e.g. when a green context or MPS leaves the call fewer SMs
  // than the device reports -- instead of waiting out the bounded waits.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, verify_kernel<P>, prob);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return SV_EUNSUPPORTED;
  if (e == cudaErrorCooperativeLaunchTooLarge) return SV_ECORESIDENT;
  return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

bool bulk_ok(const void* base, int64_t stride_bytes, int64_t row_bytes) {
  return base != nullptr && (reinterpret_cast<uintptr_t>(base) & 15) == 0 &&
         (stride_bytes & 15) == 0 && (row_bytes & 15) == 0;
}

sv_status launch_topk(const TopkPass& t, int grid, cudaStream_t stream) {
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sizeof(TopkShared))) != cudaSuccess)
    return SV_ECUDA;
  // programmatic stream serialisation, as for the persistent kernel: the
  // pass waits for the preceding work itself
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max(grid, 1)));
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = sizeof(TopkShared);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel, t);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return SV_EUNSUPPORTED;
  return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

// Geometry of a tree call on the cluster walk (sv_treewalk.cuh): the
// smallest power-of-two cluster whose slices are at most 16 KB (more CTAs
// per request would only add barriers), and the shared memory of the row
// cache and the two residual slices; ok == false when that does not fit
// (then the streaming engine takes the call).
struct TreeWalkPlan {
  bool ok = false;
  int CL = 1, Ls = 0, slot_bytes = 0;
  size_t smem = 0;
};

TreeWalkPlan tree_walk_plan(int64_t V, int es) {
  TreeWalkPlan w;
  const int64_t E = 16 / es;
  int CL = 1;
  while (CL < kTwMaxCl && ((V + CL - 1) / CL) * es > 16 * 1024) CL *= 2;
  const int64_t Ls = ((V + CL - 1) / CL + E - 1) / E * E;
  const int64_t slot = (Ls * es + 127) / 128 * 128;
  const int64_t smem = kTwSlots * slot + 2 * ((Ls + 31) / 32 * 32) * 4;
  if (smem > 200 * 1024) return w;
  w.ok = true;
  w.CL = CL;
  w.Ls = static_cast<int>(Ls);
  w.slot_bytes = static_cast<int>(slot);
  w.smem = static_cast<size_t>(smem);
  return w;
}

template <int ES>
sv_status launch_tree_walk(const TreeWalkProblem& p, const TreeWalkPlan& wp, cudaStream_t stream) {
  if (cudaFuncSetAttribute(tree_walk_kernel<ES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(wp.smem)) != cudaSuccess)
    return SV_ECUDA;
  if (wp.CL > 8 && cudaFuncSetAttribute(tree_walk_kernel<ES>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                       cudaSuccess)
    return SV_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(wp.CL));
  cfg.blockDim = dim3(kTwThreads);
  cfg.dynamicSmemBytes = wp.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(wp.CL);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int maxc = 0;
  if (cudaOccupancyMaxActiveClusters(&maxc, tree_walk_kernel<ES>, &cfg) != cudaSuccess || maxc < 1)
    return SV_ECUDA;
  const int clusters = std::min(maxc, p.B);
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * wp.CL));
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tree_walk_kernel<ES>, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return SV_EUNSUPPORTED;
  return e == cudaSuccess ? SV_OK : SV_ECUDA;
}

// The top-k pass of a chain call's filtered requests: every filtered row
// reduced to its top-k (logit, id) list and (m, Z) in the workspace's
// scratch region (layout TL).
sv_status run_topk_pass(const sv_chain_args* a, void* workspace, const Layout& L,
                        const TopkLayout& TL, const DeviceInfo& dev, cudaStream_t st) {
  const int es = es_of(a->dtype);
  char* scratch = static_cast<char*>(workspace) + L.scratch;
  TopkPass t;
  t.n_req = a->B;
  t.K = a->K;
  t.V = a->V;
  t.es = es;
  t.max_topk = a->max_top_k;
  t.seg_len = TL.seg_len;
  // the row's group maxima must fit one map of shared memory: groups of
  // 16 f tokens, f doubled until they do (one key of es bytes per group)
  t.fold = 1;
  t.group_shift = 4;
  while ((static_cast<int64_t>(a->V) + 16 * t.fold - 1) / (16 * t.fold) * es > kTkMapBytes) {
    t.fold *= 2;
    ++t.group_shift;
  }
  t.n_groups = static_cast<int>((static_cast<int64_t>(a->V) + 16 * t.fold - 1) / (16 * t.fold));
  t.has_draft = a->draft_logits != nullptr;
  t.target = static_cast<const char*>(a->target_logits);
  t.t_stride = a->target_row_stride * es;
  t.draft = static_cast<const char*>(a->draft_logits);
  t.d_stride = a->draft_logits ? a->draft_row_stride * es : 0;
  t.bulk = bulk_ok(a->target_logits, t.t_stride, static_cast<int64_t>(a->V) * es) &&
           (a->draft_logits == nullptr ||
            bulk_ok(a->draft_logits, t.d_stride, static_cast<int64_t>(a->V) * es));
  t.num_drafts = a->num_drafts;
  t.temperature = a->temperature;
  t.top_k = a->top_k;
  t.lists = reinterpret_cast<float2*>(scratch + TL.lists);
  t.mz = reinterpret_cast<float2*>(scratch + TL.mz);
  t.err = &ws_view(workspace, L).hdr->error;
  // one CTA per row at a time, every CTA resident
  const int64_t rows = static_cast<int64_t>(a->B) * (2 * a->K + 1);
  const int64_t ctas = std::min<int64_t>(rows, static_cast<int64_t>(kTkCtasPerSm) * dev.sms);
  return launch_topk(t, static_cast<int>(ctas), st);
}

__global__ void wait_selftest_kernel(WsHeader* hdr, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives: the bounded wait must give up and report
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) record_error(&hdr->error, SV_DERR_TIMEOUT);
  }
}

}  // namespace

// ------------------------------------------------- allocation-free scratch

// Callers that cannot pass a workspace -- no device allocator at hand where
// they call, or a call site where allocating device memory is not allowed or
// could block -- get this per-device array instead.  It is reserved when the
// module loads; the entry point below only looks up its address and never
// allocates.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SV_NOALLOC_SCRATCH_BYTES];

namespace {

// What the library knows about the scratch of one device: the context it
// was zeroed in (and its address there).  After a device reset or a new
// primary context the module is loaded again; the array is then looked up
// and zeroed again before its first use, so no stale address is ever used.
struct NoallocSlot {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
  bool zeroed = false;
};
NoallocSlot g_noalloc[64];

// The driver's unique id of the current context (0 when it cannot be read):
// cuCtxGetCurrent and cuCtxGetId, resolved through the runtime, so the
// library needs no link against the driver library.
unsigned long long current_ctx_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {  // under g_mu
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrent>(f1);
      get_id = reinterpret_cast<GetId>(f2);
    }
    resolved = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The scratch of the current device.  Its address is looked up on every
// call (cudaGetSymbolAddress allocates nothing); the first call in a
// context zeroes it on `stream`, ahead of whatever follows there.
sv_status noalloc_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
  if (dev < 0 || dev >= 64) return SV_EUNSUPPORTED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SV_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  const unsigned long long id = current_ctx_id();
  NoallocSlot& sl = g_noalloc[dev];
  if (!sl.zeroed || sl.ctx_id != id || sl.ptr != p) {
    if (cudaMemsetAsync(p, 0, SV_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess) return SV_ECUDA;
    sl.zeroed = true;
    sl.ctx_id = id;
    sl.ptr = p;
  }
  *out = p;
  return SV_OK;
}

}  // namespace

// Tracing (a build with -DSV_NVTX): every entry point that enqueues device
// work opens an NVTX range named after it on the calling host thread, so a
// timeline profiler shows where each call's launches were enqueued.  The
// header-only NVTX library stays inert unless a profiler attaches.
#ifdef SV_NVTX
struct SvRange {
  explicit SvRange(const char* name) { nvtxRangePushA(name); }
  ~SvRange() { nvtxRangePop(); }
};
#define SV_RANGE(name) const SvRange sv_range_(name)
#else
#define SV_RANGE(name) static_cast<void>(0)
#endif

extern "C" {

int32_t sv_version(void) { return 100; }

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK";
    case SV_EINVAL: return "SV_EINVAL: invalid argument";
    case SV_ECUDA: return "SV_ECUDA: CUDA runtime error";
    case SV_ETIMEOUT: return "SV_ETIMEOUT: a bounded device wait expired";
    case SV_EDATA: return "SV_EDATA: input data broke a precondition";
    case SV_EWORKSPACE: return "SV_EWORKSPACE: workspace missing, too small or misaligned";
    case SV_EUNSUPPORTED: return "SV_EUNSUPPORTED: needs an sm_103 (GB300) device";
    case SV_ECORESIDENT:
      return "SV_ECORESIDENT: the kernel's CTAs cannot all be resident at once on this device";
  }
  return "unknown sv_status";
}

size_t sv_chain_workspace_bytes(int32_t B, int32_t K, int32_t V, sv_dtype dtype,
                                int32_t max_top_k) {
  if (B < 0 || B > SV_MAX_B || K < 0 || K > SV_MAX_K || V < 1 || V > SV_MAX_V ||
      (dtype != SV_BF16 && dtype != SV_FP32) || max_top_k < 0 || max_top_k > SV_MAX_TOPK)
    return 0;
  return chain_layout(B, K, V, dtype, max_top_k).total;
}

size_t sv_tree_workspace_bytes(int32_t B, int32_t N, int32_t M, int32_t V, sv_dtype dtype,
                               int32_t max_top_k) {
  if (B < 0 || B > SV_MAX_TREE_B || N < 1 || N > SV_MAX_TREE_NODES || M < 1 ||
      M > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_V || (dtype != SV_BF16 && dtype != SV_FP32) ||
      max_top_k < 0 || max_top_k > SV_MAX_TOPK)
    return 0;
  return tree_layout(B, N, M, V, dtype).total;
}

sv_status sv_workspace_init(void* workspace, size_t ws_bytes, sv_stream_t stream) {
  SV_RANGE("sv_workspace_init");
  if (workspace == nullptr || ws_bytes < sizeof(WsHeader)) return SV_EWORKSPACE;
  return cudaMemsetAsync(workspace, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SV_OK
             : SV_ECUDA;
}

sv_status sv_verify_chain(const sv_chain_args* a, void* workspace, size_t ws_bytes,
                          sv_stream_t stream) {
  SV_RANGE("sv_verify_chain");
  if (a == nullptr) return SV_EINVAL;
  if (a->B < 0 || a->B > SV_MAX_B || a->K < 0 || a->K > SV_MAX_K || a->V < 1 ||
      a->V > SV_MAX_V || (a->dtype != SV_BF16 && a->dtype != SV_FP32) || a->max_top_k < 0 ||
      a->max_top_k > SV_MAX_TOPK)
    return SV_EINVAL;
  if (a->B == 0) return SV_OK;
  if (a->target_logits == nullptr || a->target_row_stride < a->V ||
      (a->draft_tokens == nullptr && a->K > 0) ||
      a->temperature == nullptr || a->uniforms == nullptr || a->out_tokens == nullptr ||
      a->out_len == nullptr || a->accept_len == nullptr)
    return SV_EINVAL;
  if (a->draft_logits != nullptr && a->draft_row_stride < a->V) return SV_EINVAL;
  const size_t need = sv_chain_workspace_bytes(a->B, a->K, a->V, a->dtype, a->max_top_k);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
      ws_bytes < need)
    return SV_EWORKSPACE;
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;

  const int es = es_of(a->dtype);
  const int chunk_el = chunk_el_of(a->dtype);
  const int ipr = (a->V + chunk_el - 1) / chunk_el;
  const Layout L = chain_layout(a->B, a->K, a->V, a->dtype, a->max_top_k);
  const TopkLayout TL = topk_layout(a->B, a->K, a->V, a->max_top_k);

  ChainProblem p;
  p.n_req = a->B;
  p.K = a->K;
  p.V = a->V;
  p.es = es;
  p.ipr = ipr;
  p.chunk_el = chunk_el;
  p.max_topk = a->max_top_k;
  p.target = static_cast<const char*>(a->target_logits);
  p.t_stride = a->target_row_stride * es;
  p.draft = static_cast<const char*>(a->draft_logits);
  p.d_stride = a->draft_logits ? a->draft_row_stride * es : 0;
  p.bulk = bulk_ok(a->target_logits, p.t_stride, static_cast<int64_t>(a->V) * es) &&
           (a->draft_logits == nullptr ||
            bulk_ok(a->draft_logits, p.d_stride, static_cast<int64_t>(a->V) * es));
  p.tokens = a->draft_tokens;
  p.num_drafts = a->num_drafts;
  p.temperature = a->temperature;
  p.top_k = a->top_k;
  p.uniforms = a->uniforms;
  p.out_tokens = a->out_tokens;
  p.out_len = a->out_len;
  p.accept_len = a->accept_len;
  p.p_at = a->p_at_draft;
  p.q_at = a->q_at_draft;
  p.ws = ws_view(workspace, L);
  p.jobs = static_cast<unsigned long long*>(p.ws.jobs);
  p.chunk2 = resid_chunk_el_of(a->dtype);
  p.ipr2 = (a->V + p.chunk2 - 1) / p.chunk2;
  char* scratch = reinterpret_cast<char*>(p.ws.scratch);
  p.topk_lists = reinterpret_cast<const float2*>(scratch + TL.lists);
  p.topk_mz = reinterpret_cast<const float2*>(scratch + TL.mz);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (a->top_k != nullptr && a->max_top_k > 0) {
    // the top-k lists first; the persistent kernel finalizes top-k
    // requests from them
    const sv_status ts = run_topk_pass(a, workspace, L, TL, dev, st);
    if (ts != SV_OK) return ts;
  }
  // control CTAs (finalizes and draw finalizes, on SMs that stream nothing):
  // three per 32 requests, 1 to 8 (at B = 64, 6 of them gave the shortest
  // step, 4 and 8 about 1.5 % longer); the rest of the grid streams.  A call with
  // top-k lists gets one per 4 requests, up to half the SMs: its filtered
  // requests finalize from the lists alone, so their finalizes are all the
  // work there is for them
  const bool with_lists = a->top_k != nullptr && a->max_top_k > 0;
  const int n_ctrl = static_cast<int>(
      with_lists ? std::min<int64_t>(std::max(1, dev.sms / 2), std::max<int64_t>(1, (a->B + 3) / 4))
                 : std::min<int64_t>(8, std::max<int64_t>(1, (3 * a->B + 31) / 32)));
  const int64_t items_max = static_cast<int64_t>(a->B) * (2 * a->K + 1) * ipr;
  const int stream_ctas = static_cast<int>(
      std::min<int64_t>(std::max<int64_t>(items_max, 1), dev.sms - n_ctrl));
  p.n_ctrl = n_ctrl;
  return launch(p, stream_ctas + n_ctrl, st);
}

sv_status sv_verify_tree(const sv_tree_args* a, void* workspace, size_t ws_bytes,
                         sv_stream_t stream) {
  SV_RANGE("sv_verify_tree");
  if (a == nullptr) return SV_EINVAL;
  if (a->B < 0 || a->B > SV_MAX_TREE_B || a->N < 1 || a->N > SV_MAX_TREE_NODES || a->M < 1 ||
      a->M > SV_MAX_TREE_NODES || a->V < 1 || a->V > SV_MAX_V || a->max_depth < 0 ||
      a->max_depth >= a->N || (a->dtype != SV_BF16 && a->dtype != SV_FP32) ||
      a->mode < SV_TREE_MSS || a->mode > SV_TREE_NAIVE || a->max_top_k < 0 ||
      a->max_top_k > SV_MAX_TOPK)
    return SV_EINVAL;
  if (a->B == 0) return SV_OK;
  if (a->target_logits == nullptr || a->target_row_stride < a->V || a->node_tokens == nullptr ||
      a->parent == nullptr || a->q_row == nullptr || a->temperature == nullptr ||
      a->u_accept == nullptr || a->u_sample == nullptr || a->out_tokens == nullptr ||
      a->out_len == nullptr || a->accept_len == nullptr || a->accepted_nodes == nullptr)
    return SV_EINVAL;
  if (a->draft_logits != nullptr && a->draft_row_stride < a->V) return SV_EINVAL;
  const size_t need = sv_tree_workspace_bytes(a->B, a->N, a->M, a->V, a->dtype, a->max_top_k);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
      ws_bytes < need)
    return SV_EWORKSPACE;
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;

  const int es = es_of(a->dtype);
  const TreeWalkPlan wp = tree_walk_plan(a->V, es);
  if (wp.ok) {
    // the cluster walk: one cluster per request, reading only the rows on
    // the path
    TreeWalkProblem w;
    w.B = a->B;
    w.N = a->N;
    w.M = a->M;
    w.V = a->V;
    w.max_depth = a->max_depth;
    w.es = es;
    w.mode = static_cast<int>(a->mode);
    w.Ls = wp.Ls;
    w.slot_bytes = wp.slot_bytes;
    w.target = static_cast<const char*>(a->target_logits);
    w.t_stride = a->target_row_stride * es;
    w.draft = static_cast<const char*>(a->draft_logits);
    w.d_stride = a->draft_logits ? a->draft_row_stride * es : 0;
    w.bulk = bulk_ok(a->target_logits, w.t_stride, static_cast<int64_t>(a->V) * es) &&
             (a->draft_logits == nullptr ||
              bulk_ok(a->draft_logits, w.d_stride, static_cast<int64_t>(a->V) * es));
    w.tokens = a->node_tokens;
    w.parent = a->parent;
    w.q_row = a->q_row;
    w.num_nodes = a->num_nodes;
    w.temperature = a->temperature;
    w.top_k = a->top_k;
    w.u_accept = a->u_accept;
    w.u_sample = a->u_sample;
    w.out_tokens = a->out_tokens;
    w.out_len = a->out_len;
    w.accept_len = a->accept_len;
    w.accepted_nodes = a->accepted_nodes;
    w.hdr = static_cast<WsHeader*>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return es == 2 ? launch_tree_walk<2>(w, wp, st) : launch_tree_walk<4>(w, wp, st);
  }
  const int chunk_el = chunk_el_of(a->dtype);
  const int ipr = (a->V + chunk_el - 1) / chunk_el;
  const Layout L = tree_layout(a->B, a->N, a->M, a->V, a->dtype);
  TreeProblem p;
  p.n_req = a->B;
  p.N = a->N;
  p.M = a->M;
  p.V = a->V;
  p.max_depth = a->max_depth;
  p.es = es;
  p.ipr = ipr;
  p.chunk_el = chunk_el;
  p.max_topk = a->max_top_k;
  p.mode = static_cast<int>(a->mode);
  p.target = static_cast<const char*>(a->target_logits);
  p.t_stride = a->target_row_stride * es;
  p.draft = static_cast<const char*>(a->draft_logits);
  p.d_stride = a->draft_logits ? a->draft_row_stride * es : 0;
  p.bulk = bulk_ok(a->target_logits, p.t_stride, static_cast<int64_t>(a->V) * es) &&
           (a->draft_logits == nullptr ||
            bulk_ok(a->draft_logits, p.d_stride, static_cast<int64_t>(a->V) * es));
  p.tokens = a->node_tokens;
  p.parent = a->parent;
  p.q_row = a->q_row;
  p.num_nodes = a->num_nodes;
  p.temperature = a->temperature;
  p.top_k = a->top_k;
  p.u_accept = a->u_accept;
  p.u_sample = a->u_sample;
  p.out_tokens = a->out_tokens;
  p.out_len = a->out_len;
  p.accept_len = a->accept_len;
  p.accepted_nodes = a->accepted_nodes;
  p.ws = ws_view(workspace, L);

  const int64_t items_max = static_cast<int64_t>(a->B) * (a->N + a->M) * ipr;
  const int grid = static_cast<int>(std::min<int64_t>(std::max<int64_t>(items_max, 1), dev.sms));
  return launch(p, grid, reinterpret_cast<cudaStream_t>(stream));
}

sv_status sv_get_error(void* workspace, sv_stream_t stream, int32_t* device_flags) {
  SV_RANGE("sv_get_error");
  if (workspace == nullptr) return SV_EWORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SV_ECUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return SV_ECUDA;
  const int zero = 0;
  if (cudaMemcpy(static_cast<char*>(workspace) + offsetof(WsHeader, error), &zero, sizeof(int),
                 cudaMemcpyHostToDevice) != cudaSuccess)
    return SV_ECUDA;
  if (device_flags) *device_flags = h.error;
  if (h.error & SV_DERR_TIMEOUT) return SV_ETIMEOUT;
  return h.error ? SV_EDATA : SV_OK;
}

sv_status sv_selftest_wait_timeout(void* workspace, size_t ws_bytes, int64_t limit_ns,
                                   sv_stream_t stream) {
  if (workspace == nullptr || ws_bytes < sizeof(WsHeader) ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return SV_EWORKSPACE;
  if (limit_ns <= 0 || limit_ns > 2000000000ll) return SV_EINVAL;
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  wait_selftest_kernel<<<1, 32, 0, s>>>(static_cast<WsHeader*>(workspace),
                                        static_cast<uint64_t>(limit_ns));
  if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;
  return sv_get_error(workspace, stream, nullptr);
}


sv_status sv_tree_mask(const sv_tree_mask_args* a, void* workspace, size_t ws_bytes,
                       sv_stream_t stream) {
  SV_RANGE("sv_tree_mask");
  if (a == nullptr) return SV_EINVAL;
  if (a->B < 0 || a->B > SV_MAX_TREE_B || a->N < 1 || a->N > SV_MAX_TREE_NODES ||
      a->words < (a->N + 31) / 32 || a->words > 1 << 20)
    return SV_EINVAL;
  if (a->B == 0) return SV_OK;
  if (a->parent == nullptr || a->mask == nullptr || a->depth == nullptr) return SV_EINVAL;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
      ws_bytes < SV_MIN_WORKSPACE_BYTES)
    return SV_EWORKSPACE;
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;
  MaskProblem p;
  p.B = a->B;
  p.N = a->N;
  p.words = a->words;
  p.parent = a->parent;
  p.num_nodes = a->num_nodes;
  p.mask = a->mask;
  p.depth = a->depth;
  p.hdr = static_cast<WsHeader*>(workspace);
  tree_mask_kernel<<<(a->B + kMaskWarps - 1) / kMaskWarps, kMaskWarps * 32, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

sv_status sv_row_stats(const sv_chain_args* a, float* alpha, float* expected, void* workspace,
                       size_t ws_bytes, sv_stream_t stream) {
  SV_RANGE("sv_row_stats");
  if (a == nullptr) return SV_EINVAL;
  if (a->B < 0 || a->B > SV_MAX_B || a->K < 0 || a->K > SV_MAX_K || a->V < 1 ||
      a->V > SV_MAX_V || (a->dtype != SV_BF16 && a->dtype != SV_FP32) || a->max_top_k < 0 ||
      a->max_top_k > SV_MAX_TOPK)
    return SV_EINVAL;
  if (a->B == 0) return SV_OK;
  if (a->target_logits == nullptr || a->target_row_stride < a->V || a->temperature == nullptr ||
      expected == nullptr)
    return SV_EINVAL;
  if (a->K > 0 && (a->draft_logits == nullptr || a->draft_row_stride < a->V || alpha == nullptr))
    return SV_EINVAL;
  const bool with_topk = a->top_k != nullptr && a->max_top_k > 0;
  const Layout L0 = layout_for(0, 0, 0);
  const size_t need =
      with_topk ? sv_chain_workspace_bytes(a->B, a->K, a->V, a->dtype, a->max_top_k) : L0.jobs;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
      ws_bytes < need)
    return SV_EWORKSPACE;
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;
  const int es = es_of(a->dtype);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (with_topk && a->K > 0) {
    // filtered sampled requests: the top-k lists, then their statistics
    const Layout L = chain_layout(a->B, a->K, a->V, a->dtype, a->max_top_k);
    const TopkLayout TL = topk_layout(a->B, a->K, a->V, a->max_top_k);
    const sv_status ts = run_topk_pass(a, workspace, L, TL, dev, s);
    if (ts != SV_OK) return ts;
    char* scratch = static_cast<char*>(workspace) + L.scratch;
    StatsTopkProblem q;
    q.B = a->B;
    q.K = a->K;
    q.V = a->V;
    q.max_topk = a->max_top_k;
    q.has_draft = true;
    q.num_drafts = a->num_drafts;
    q.temperature = a->temperature;
    q.top_k = a->top_k;
    q.lists = reinterpret_cast<float2*>(scratch + TL.lists);
    q.mz = reinterpret_cast<float2*>(scratch + TL.mz);
    q.alpha = alpha;
    q.expected = expected;
    q.hdr = static_cast<WsHeader*>(workspace);
    // programmatic stream serialisation: the kernel waits for the top-k pass
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((a->B + kStTkWarps - 1) / kStTkWarps));
    cfg.blockDim = dim3(kStTkWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, row_stats_topk_kernel, q) != cudaSuccess) return SV_ECUDA;
  }
  StatsProblem p;
  p.B = a->B;
  p.K = a->K;
  p.V = a->V;
  p.max_topk = with_topk ? a->max_top_k : 0;
  p.target = static_cast<const char*>(a->target_logits);
  p.t_stride = a->target_row_stride * es;
  p.draft = a->K > 0 ? static_cast<const char*>(a->draft_logits) : p.target;
  p.d_stride = a->K > 0 ? a->draft_row_stride * es : p.t_stride;
  p.vec = bulk_ok(p.target, p.t_stride, static_cast<int64_t>(a->V) * es) &&
          bulk_ok(p.draft, p.d_stride, static_cast<int64_t>(a->V) * es);
  p.num_drafts = a->num_drafts;
  p.temperature = a->temperature;
  p.top_k = a->top_k;
  p.alpha = alpha;
  p.expected = expected;
  p.hdr = static_cast<WsHeader*>(workspace);
  p.tickets = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + L0.tickets);
  const unsigned grid = static_cast<unsigned>(a->B) * static_cast<unsigned>(std::max(a->K, 1)) *
                        static_cast<unsigned>(kStCluster);
  if (es == 2) row_stats_kernel<2><<<grid, kStThreads, 0, s>>>(p);
  else row_stats_kernel<4><<<grid, kStThreads, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

sv_status sv_verify_chain_noalloc(const sv_chain_args* a, sv_stream_t stream) {
  SV_RANGE("sv_verify_chain_noalloc");
  if (a == nullptr) return SV_EINVAL;
  if (a->B == 0) return sv_verify_chain(a, nullptr, 0, stream);
  const size_t need = sv_chain_workspace_bytes(a->B, a->K, a->V, a->dtype, a->max_top_k);
  if (need == 0) return SV_EINVAL;
  if (need > SV_NOALLOC_SCRATCH_BYTES) return SV_EWORKSPACE;  // too large for the scratch
  DeviceInfo dev;
  const sv_status ds = device_info(dev);
  if (ds != SV_OK) return ds;
  void* ws = nullptr;
  const sv_status st = noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &ws);
  if (st != SV_OK) return st;
  return sv_verify_chain(a, ws, SV_NOALLOC_SCRATCH_BYTES, stream);
}

sv_status sv_noalloc_get_error(sv_stream_t stream, int32_t* device_flags) {
  SV_RANGE("sv_noalloc_get_error");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const sv_status st = noalloc_scratch(s, &ws);
  if (st != SV_OK) return st;
  const sv_status es = sv_get_error(ws, stream, device_flags);
  if (es == SV_EDATA || es == SV_ETIMEOUT) {
    // a failed call may leave counters set: start the next one from zero
    if (cudaMemsetAsync(ws, 0, SV_NOALLOC_SCRATCH_BYTES, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return SV_ECUDA;
  }
  return es;
}

}  // extern "C"
