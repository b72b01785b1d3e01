// C ABI of the swin_wattn library: argument validation, plan ownership, launches and
// error surfacing. No exception, abort or trap crosses this boundary.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>

#include "common.cuh"

namespace swin {
cudaError_t launch_bias_tables(const Plan& p, const float* table, bool with_mask, cudaStream_t st);
bool fwd_fp8_applies(const Plan& pl);
cudaError_t fwd_fp8_launch(const Plan& pl, const void* qkv8, float sq, float sk, float sv, void* out,
                           cudaStream_t st);
cudaError_t launch_build_mask(int H, int W, int M, int s, float* mask, cudaStream_t st);
cudaError_t launch_gather_map(int H, int W, int M, int s, int32_t* out, cudaStream_t st);
cudaError_t launch_relidx(int M, int32_t* out, cudaStream_t st);
size_t tc_tables_bytes(const Plan& pl);
cudaError_t launch_tc_tables(const Plan& pl, cudaStream_t st);
size_t bias_frag_bytes(int M, int nH);
size_t mask_frag_bytes(int M);
cudaError_t fwd_config(const Plan& pl, FwdLaunch* L);
cudaError_t fwd_launch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out,
                       cudaStream_t st);
cudaError_t fwd_launch_batch(const Plan& pl, const FwdLaunch& L, const void* qkv, void* out,
                             int batch, cudaStream_t st);
cudaError_t bwd_config(const Plan& pl, BwdLaunch* L);
bool bwd_tc_applies(const Plan& pl);
cudaError_t bwd_tc_config(const Plan& pl, BwdLaunch* L);
cudaError_t qkv_proj_launch(const void* x, const float* gamma, const float* beta, const void* w, const float* b,
                            void* out, int T, int C, float eps, void* workspace, int* status, cudaStream_t st);
size_t qkv_workspace_bytes(int C, int64_t T);
size_t qkv_prepared_bytes(int C);
size_t qkv_stats_bytes(int64_t T);
cudaError_t qkv_prepare_launch(const float* gamma, const float* beta, const void* w, const float* b, int C,
                               void* prepared, cudaStream_t st);
cudaError_t qkv_proj_prepared_launch(const void* x, const void* prepared, void* out, int T, int C, float eps,
                                     void* stats_workspace, int* status, cudaStream_t st);
int qkv_launches(int T, int C, bool fold);
cudaError_t qkv_proj_fp8_launch(const void* x, const void* prepared, void* out8, int T, int C, float eps,
                                const float scales[3], unsigned int* amax, void* stats_workspace, int* status,
                                cudaStream_t st);
cudaError_t proj_residual_launch(const void* o, const void* wp, const float* bp, const void* residual, void* y,
                                 int T, int C, int* status, cudaStream_t st);
cudaError_t bwd_launch(const Plan& pl, const BwdLaunch& L, const void* qkv, const void* dout,
                       void* dqkv, float* dtable, cudaStream_t st);
}  // namespace swin

// Streams and events of the host-buffer forward's copy/compute pipeline, created on
// its first use.
constexpr int kHostChunks = 4;
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kHostChunks] = {}, computed[kHostChunks] = {};
};

struct swin_wattn_plan_s {
  swin::Plan p;
  swin::FwdLaunch fwd;
  swin::BwdLaunch bwd;
  HostPipe pipe;
};

namespace {

thread_local char g_last_error[256] = "";
thread_local uint64_t g_launches = 0;

int cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return SWIN_WATTN_ERR_CUDA;
}

// A pointer the GPU can dereference: device or managed memory, or host memory mapped
// into the device address space.
int check_device_ptr(const void* ptr, size_t align) {
  if (ptr == nullptr) return SWIN_WATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ptr) % align != 0) return SWIN_WATTN_ERR_MISALIGNED;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return SWIN_WATTN_OK;
  if (a.type == cudaMemoryTypeHost && a.devicePointer == ptr) return SWIN_WATTN_OK;
  return SWIN_WATTN_ERR_INVALID_ARG;
}

// Live plans. A handle is checked against this set before it is dereferenced, so a
// destroyed or foreign handle is reported instead of read.
std::mutex g_plans_mu;
std::unordered_set<const swin_wattn_plan_s*> g_plans;

int check_plan(const swin_wattn_plan_s* pl) {
  if (pl == nullptr) return SWIN_WATTN_ERR_BAD_PLAN;
  {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    if (g_plans.find(pl) == g_plans.end()) return SWIN_WATTN_ERR_BAD_PLAN;
  }
  if (pl->p.magic != swin::kPlanMagic) return SWIN_WATTN_ERR_BAD_PLAN;
  return SWIN_WATTN_OK;
}

void free_pipe(HostPipe& hp) {
  if (!hp.ready) return;
  for (int c = 0; c < kHostChunks; ++c) {
    cudaEventDestroy(hp.loaded[c]);
    cudaEventDestroy(hp.computed[c]);
  }
  cudaEventDestroy(hp.start);
  cudaEventDestroy(hp.done);
  cudaStreamDestroy(hp.in);
  cudaStreamDestroy(hp.out);
  hp.ready = false;
}

void free_plan_buffers(swin::Plan& p) {
  if (p.dense_bias) cudaFree(p.dense_bias);
  if (p.mask) cudaFree(p.mask);
  if (p.dt_partial) cudaFree(p.dt_partial);
  if (p.bias_frag) cudaFree(p.bias_frag);
  if (p.mask_frag) cudaFree(p.mask_frag);
  if (p.err) cudaFree(p.err);
  if (p.tc_tables) cudaFree(p.tc_tables);

  p.dense_bias = p.mask = p.dt_partial = nullptr;
  p.bias_frag = nullptr;
  p.mask_frag = nullptr;
  p.err = nullptr;
  p.tc_tables = nullptr;
}

}  // namespace

namespace swin {
void set_last_error(const char* msg) { std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
int check_device_ptr_abi(const void* ptr, size_t align) { return check_device_ptr(ptr, align); }
// Kernel launches issued by the calling thread outside this file (swin_wattn_launch_count).
void count_launches(int n) { g_launches += (uint64_t)n; }

namespace {
std::atomic<uint64_t> g_wait_ns{1000000000ull};
std::atomic<int> g_fault{kFaultNone};
}  // namespace
uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int fault_site() { return g_fault.load(std::memory_order_relaxed); }
}  // namespace swin

#ifdef SWIN_WATTN_FAULT_INJECTION
#include "../../include/swin_wattn_debug.h"

extern "C" int swin_wattn_debug_set_fault(int site, int64_t wait_limit_ns) {
  if (site < swin::kFaultNone || site > swin::kFaultGemm) return SWIN_WATTN_ERR_INVALID_ARG;
  if (wait_limit_ns < 1000 || wait_limit_ns > 10000000000ll) return SWIN_WATTN_ERR_INVALID_ARG;
  swin::g_wait_ns.store((uint64_t)wait_limit_ns);
  swin::g_fault.store(site);
  return SWIN_WATTN_OK;
}
#endif

extern "C" {

const char* swin_wattn_status_string(int status) {
  switch (status) {
    case SWIN_WATTN_OK: return "ok";
    case SWIN_WATTN_ERR_INVALID_ARG: return "invalid argument";
    case SWIN_WATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case SWIN_WATTN_ERR_MISALIGNED: return "misaligned pointer";
    case SWIN_WATTN_ERR_BAD_PLAN: return "bad plan handle";
    case SWIN_WATTN_ERR_CUDA: return "CUDA error";
    case SWIN_WATTN_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* swin_wattn_last_error(void) { return g_last_error; }

uint64_t swin_wattn_launch_count(int reset) {
  const uint64_t n = g_launches;
  if (reset) g_launches = 0;
  return n;
}

int swin_wattn_plan(swin_wattn_plan_t* out, int B, int H, int W, int C, int num_heads,
                    int window, int shift, int dtype, const float* bias_table,
                    struct CUstream_st* stream) {
  if (out == nullptr) return SWIN_WATTN_ERR_INVALID_ARG;
  *out = nullptr;
  if (B < 0 || H <= 0 || W <= 0 || C <= 0 || num_heads <= 0) return SWIN_WATTN_ERR_INVALID_ARG;
  if (dtype != SWIN_WATTN_BF16 && dtype != SWIN_WATTN_FP32) return SWIN_WATTN_ERR_INVALID_ARG;
  if (window != 4 && window != 7 && window != 12) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (shift < 0 || shift >= window) return SWIN_WATTN_ERR_INVALID_ARG;
  if (H % window != 0 || W % window != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (C % num_heads != 0 || C / num_heads != swin::kHeadDim) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * H * W * 3 * C >= ((int64_t)1 << 40)) return SWIN_WATTN_ERR_UNSUPPORTED;
  int rc = check_device_ptr(bias_table, 4);
  if (rc != SWIN_WATTN_OK) return rc;

  swin_wattn_plan_s* pl = new (std::nothrow) swin_wattn_plan_s();
  if (pl == nullptr) return SWIN_WATTN_ERR_INVALID_ARG;
  swin::Plan& p = pl->p;
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = H;
  p.W = W;
  p.C = C;
  p.nH = num_heads;
  p.M = window;
  p.s = shift;
  p.dtype = dtype;
  p.N = window * window;
  p.nWy = H / window;
  p.nWx = W / window;
  p.nW = p.nWy * p.nWx;

  cudaError_t e = cudaGetDevice(&p.device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, p.device);
  const size_t nn = (size_t)p.N * p.N;
  if (e == cudaSuccess) e = cudaMalloc(&p.dense_bias, sizeof(float) * nn * p.nH);
  // The mask tensor always exists (all zeros for s = 0) so that it can be dumped.
  if (e == cudaSuccess) e = cudaMalloc(&p.mask, sizeof(float) * nn * p.nW);
  if (e == cudaSuccess) e = cudaMalloc(&p.bias_frag, swin::bias_frag_bytes(p.M, p.nH));
  if (e == cudaSuccess && p.s > 0) e = cudaMalloc(&p.mask_frag, swin::mask_frag_bytes(p.M));
  if (e == cudaSuccess) e = cudaMalloc(&p.err, sizeof(int));
  if (e == cudaSuccess && swin::tc_tables_bytes(p) > 0) e = cudaMalloc(&p.tc_tables, swin::tc_tables_bytes(p));
  if (e == cudaSuccess) e = cudaMemsetAsync(p.err, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream));

  if (e == cudaSuccess) e = swin::fwd_config(p, &pl->fwd);
  if (e == cudaSuccess) e = swin::bwd_config(p, &pl->bwd);
  // the table-gradient partials, sized for either backward kernel (the choice may change)
  int partial_rows = pl->bwd.partial_rows;
  if (e == cudaSuccess && swin::bwd_tc_applies(p)) {
    swin::BwdLaunch Lt;
    e = swin::bwd_tc_config(p, &Lt);
    if (e == cudaSuccess && Lt.partial_rows > partial_rows) partial_rows = Lt.partial_rows;
  }
  if (e == cudaSuccess && partial_rows > 0) {
    p.dt_partial_rows = partial_rows;
    e = cudaMalloc(&p.dt_partial, sizeof(float) * (size_t)p.dt_partial_rows * (2 * p.M - 1) *
                                      (2 * p.M - 1));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (e == cudaSuccess) {
    e = swin::launch_bias_tables(p, bias_table, true, st);
    ++g_launches;
  }
  if (e == cudaSuccess) {
    e = swin::launch_build_mask(p.H, p.W, p.M, p.s, p.mask, st);
    ++g_launches;
  }
  p.tc_stale = p.tc_tables != nullptr;  // built before the first tcgen05 forward
  if (e != cudaSuccess) {
    rc = cuda_fail(e, "swin_wattn_plan");
    free_plan_buffers(p);
    delete pl;
    return rc;
  }
  p.magic = swin::kPlanMagic;
  {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    g_plans.insert(pl);
  }
  *out = pl;
  return SWIN_WATTN_OK;
}

int swin_wattn_set_bias(swin_wattn_plan_t plan, const float* bias_table,
                        struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  rc = check_device_ptr(bias_table, 4);
  if (rc != SWIN_WATTN_OK) return rc;
  swin::Plan& p = plan->p;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // One launch: the mma fragments and the dense bias, both from the table. The tcgen05
  // tables are rebuilt before the next forward that uses them.
  cudaError_t e = swin::launch_bias_tables(p, bias_table, false, st);
  ++g_launches;
  p.tc_stale = p.tc_tables != nullptr;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_set_bias");
}

// The tcgen05 forward's constant tables, rebuilt from the dense bias on `st` when the bias
// changed since they were last built.
static cudaError_t ensure_tc_tables(swin_wattn_plan_s* plan, cudaStream_t st, bool for_bwd = false) {
  swin::Plan& p = plan->p;
  if (!(for_bwd ? plan->bwd.tc : plan->fwd.tc) || !p.tc_stale) return cudaSuccess;
  const cudaError_t e = swin::launch_tc_tables(p, st);
  ++g_launches;
  if (e == cudaSuccess) p.tc_stale = false;
  return e;
}

int swin_wattn_fwd(swin_wattn_plan_t plan, const void* qkv, void* out,
                   struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  const swin::Plan& p = plan->p;
  if (p.B == 0) return SWIN_WATTN_OK;
  if ((rc = check_device_ptr(qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(out, 16)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = ensure_tc_tables(plan, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = swin::fwd_launch(p, plan->fwd, qkv, out, reinterpret_cast<cudaStream_t>(stream));
  ++g_launches;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_fwd");
}

int swin_wattn_fwd_fp8(swin_wattn_plan_t plan, const void* qkv8, float scale_q, float scale_k, float scale_v,
                       void* out, struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  const swin::Plan& p = plan->p;
  if (!swin::fwd_fp8_applies(p)) return SWIN_WATTN_ERR_UNSUPPORTED;
  for (const float sc : {scale_q, scale_k, scale_v})
    if (!(sc > 0.0f) || !std::isfinite(sc)) return SWIN_WATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale_q * scale_k) || !(scale_q * scale_k > 0.0f)) return SWIN_WATTN_ERR_INVALID_ARG;
  if (p.B == 0) return SWIN_WATTN_OK;
  if ((rc = check_device_ptr(qkv8, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(out, 16)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = swin::fwd_fp8_launch(p, qkv8, scale_q, scale_k, scale_v, out, reinterpret_cast<cudaStream_t>(stream));
  ++g_launches;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_fwd_fp8");
}

int swin_wattn_fwd_host(swin_wattn_plan_t plan, const void* qkv_host, void* out_host,
                        void* dev_qkv, void* dev_out, struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  const swin::Plan& p = plan->p;
  if (p.B == 0) return SWIN_WATTN_OK;
  if (qkv_host == nullptr || out_host == nullptr) return SWIN_WATTN_ERR_INVALID_ARG;
  if ((rc = check_device_ptr(dev_qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(dev_out, 16)) != SWIN_WATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = ensure_tc_tables(plan, st);
  if (e != cudaSuccess) return cuda_fail(e, "swin_wattn_fwd_host");
  HostPipe& hp = plan->pipe;
  if (!hp.ready) {
    e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
    for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
      e = cudaEventCreateWithFlags(&hp.loaded[c], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.computed[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e, "swin_wattn_fwd_host");
    hp.ready = true;
  }
  // Batch chunks flow through three queues: copy-in, compute (the caller's stream) and
  // copy-out, so the two copy directions and the kernels overlap; the caller's stream
  // finally waits for the last copy-out, keeping the call ordered on `stream`.
  const size_t esz = p.dtype == SWIN_WATTN_FP32 ? 4 : 2;
  const size_t img_in = (size_t)p.H * p.W * 3 * p.C * esz, img_out = (size_t)p.H * p.W * p.C * esz;
  const int nchunk = p.B < kHostChunks ? p.B : kHostChunks;
  e = cudaEventRecord(hp.start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.in, hp.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.out, hp.start, 0);
  for (int c = 0; c < nchunk && e == cudaSuccess; ++c) {
    const int b0 = (int)((int64_t)p.B * c / nchunk), b1 = (int)((int64_t)p.B * (c + 1) / nchunk);
    const size_t n_in = img_in * (b1 - b0), n_out = img_out * (b1 - b0);
    const char* hsrc = static_cast<const char*>(qkv_host) + img_in * b0;
    char* dq = static_cast<char*>(dev_qkv) + img_in * b0;
    char* dout = static_cast<char*>(dev_out) + img_out * b0;
    e = cudaMemcpyAsync(dq, hsrc, n_in, cudaMemcpyHostToDevice, hp.in);
    if (e == cudaSuccess) e = cudaEventRecord(hp.loaded[c], hp.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp.loaded[c], 0);
    if (e == cudaSuccess) {
      e = swin::fwd_launch_batch(p, plan->fwd, dq, dout, b1 - b0, st);
      ++g_launches;
    }
    if (e == cudaSuccess) e = cudaEventRecord(hp.computed[c], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp.out, hp.computed[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(out_host) + img_out * b0, dout, n_out,
                          cudaMemcpyDeviceToHost, hp.out);
  }
  if (e == cudaSuccess) e = cudaEventRecord(hp.done, hp.out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, hp.done, 0);
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_fwd_host");
}

int swin_wattn_bwd(swin_wattn_plan_t plan, const void* qkv, const void* dout, void* dqkv,
                   float* dtable, struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  const swin::Plan& p = plan->p;
  if (plan->bwd.grid == 0 && p.B > 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((rc = check_device_ptr(dtable, 4)) != SWIN_WATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t tbytes = sizeof(float) * (size_t)(2 * p.M - 1) * (2 * p.M - 1) * p.nH;
  if (p.B == 0) {
    cudaError_t e = cudaMemsetAsync(dtable, 0, tbytes, st);
    return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_bwd");
  }
  if ((rc = check_device_ptr(qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(dout, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(dqkv, 16)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = ensure_tc_tables(plan, st, true);
  if (e == cudaSuccess) e = swin::bwd_launch(p, plan->bwd, qkv, dout, dqkv, dtable, st);
  g_launches += 2;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_bwd");
}

int swin_wattn_debug_maps(swin_wattn_plan_t plan, int32_t* gather, int32_t* relidx,
                          float* mask, float* dense_bias, struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  const swin::Plan& p = plan->p;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t nn = (size_t)p.N * p.N;
  cudaError_t e = cudaSuccess;
  if (gather) {
    if ((rc = check_device_ptr(gather, 4)) != SWIN_WATTN_OK) return rc;
    e = swin::launch_gather_map(p.H, p.W, p.M, p.s, gather, st);
    ++g_launches;
  }
  if (e == cudaSuccess && relidx) {
    if ((rc = check_device_ptr(relidx, 4)) != SWIN_WATTN_OK) return rc;
    e = swin::launch_relidx(p.M, relidx, st);
    ++g_launches;
  }
  if (e == cudaSuccess && mask) {
    if ((rc = check_device_ptr(mask, 4)) != SWIN_WATTN_OK) return rc;
    e = cudaMemcpyAsync(mask, p.mask, sizeof(float) * nn * p.nW, cudaMemcpyDeviceToDevice, st);
  }
  if (e == cudaSuccess && dense_bias) {
    if ((rc = check_device_ptr(dense_bias, 4)) != SWIN_WATTN_OK) return rc;
    e = cudaMemcpyAsync(dense_bias, p.dense_bias, sizeof(float) * nn * p.nH,
                        cudaMemcpyDeviceToDevice, st);
  }
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_debug_maps");
}

size_t swin_wattn_qkv_workspace_bytes(int C, int tokens) {
  return (C < 32 || C > 1536 || C % 32 != 0 || tokens < 0) ? 0 : swin::qkv_workspace_bytes(C, tokens);
}

int swin_wattn_qkv_proj(const void* x, const float* gamma, const float* beta, const void* w_qkv,
                        const float* b_qkv, void* qkv, int tokens, int C, float eps, void* workspace,
                        size_t workspace_bytes, int* status, struct CUstream_st* stream) {
  if (tokens < 0 || !(eps >= 0.0f) || !std::isfinite(eps)) return SWIN_WATTN_ERR_INVALID_ARG;
  if (C < 32 || C > 1536 || C % 32 != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)tokens >= ((int64_t)1 << 31)) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (tokens == 0) return SWIN_WATTN_OK;
  if (workspace_bytes < swin::qkv_workspace_bytes(C, tokens)) {
    swin::set_last_error("swin_wattn_qkv_proj: workspace smaller than swin_wattn_qkv_workspace_bytes(C, tokens)");
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = check_device_ptr(x, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(w_qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(workspace, 256)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(gamma, 4)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(beta, 4)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(b_qkv, 4)) != SWIN_WATTN_OK) return rc;
  if (status != nullptr && (rc = check_device_ptr(status, 4)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = swin::qkv_proj_launch(x, gamma, beta, w_qkv, b_qkv, qkv, tokens, C, eps, workspace, status,
                                        reinterpret_cast<cudaStream_t>(stream));
  g_launches += 2;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_qkv_proj");
}

size_t swin_wattn_qkv_prepared_bytes(int C) {
  return (C < 32 || C > 1536 || C % 32 != 0) ? 0 : swin::qkv_prepared_bytes(C);
}

size_t swin_wattn_qkv_stats_bytes(int tokens) { return tokens < 0 ? 0 : swin::qkv_stats_bytes(tokens); }

int swin_wattn_qkv_prepare(const float* gamma, const float* beta, const void* w_qkv, const float* b_qkv, int C,
                           void* prepared, size_t prepared_bytes, struct CUstream_st* stream) {
  if (C < 32 || C > 1536 || C % 32 != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (prepared_bytes < swin::qkv_prepared_bytes(C)) {
    swin::set_last_error("swin_wattn_qkv_prepare: buffer smaller than swin_wattn_qkv_prepared_bytes(C)");
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = check_device_ptr(w_qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(prepared, 256)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(gamma, 4)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(beta, 4)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(b_qkv, 4)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = swin::qkv_prepare_launch(gamma, beta, w_qkv, b_qkv, C, prepared,
                                           reinterpret_cast<cudaStream_t>(stream));
  ++g_launches;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_qkv_prepare");
}

int swin_wattn_qkv_proj_prepared(const void* x, const void* prepared, void* qkv, int tokens, int C, float eps,
                                 void* stats_workspace, size_t stats_bytes, int* status, struct CUstream_st* stream) {
  if (tokens < 0 || !(eps >= 0.0f) || !std::isfinite(eps)) return SWIN_WATTN_ERR_INVALID_ARG;
  if (C < 32 || C > 1536 || C % 32 != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)tokens >= ((int64_t)1 << 31)) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (tokens == 0) return SWIN_WATTN_OK;
  if (stats_bytes < swin::qkv_stats_bytes(tokens)) {
    swin::set_last_error("swin_wattn_qkv_proj_prepared: statistics workspace smaller than "
                         "swin_wattn_qkv_stats_bytes(tokens)");
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = check_device_ptr(x, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(prepared, 256)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(qkv, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(stats_workspace, 16)) != SWIN_WATTN_OK) return rc;
  if (status != nullptr && (rc = check_device_ptr(status, 4)) != SWIN_WATTN_OK) return rc;
  cudaError_t e = swin::qkv_proj_prepared_launch(x, prepared, qkv, tokens, C, eps, stats_workspace, status,
                                                 reinterpret_cast<cudaStream_t>(stream));
  g_launches += swin::qkv_launches(tokens, C, false);
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_qkv_proj_prepared");
}

int swin_wattn_qkv_proj_prepared_fp8(const void* x, const void* prepared, void* qkv8, int tokens, int C, float eps,
                                     float scale_q, float scale_k, float scale_v, float* amax, void* stats_workspace,
                                     size_t stats_bytes, int* status, struct CUstream_st* stream) {
  if (tokens < 0 || !(eps >= 0.0f) || !std::isfinite(eps)) return SWIN_WATTN_ERR_INVALID_ARG;
  for (const float sc : {scale_q, scale_k, scale_v})
    if (!(sc > 0.0f) || !std::isfinite(sc) || !std::isfinite(1.0f / sc)) return SWIN_WATTN_ERR_INVALID_ARG;
  if (C < 32 || C > 1536 || C % 32 != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)tokens >= ((int64_t)1 << 31)) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (tokens == 0) return SWIN_WATTN_OK;
  if (stats_bytes < swin::qkv_stats_bytes(tokens)) {
    swin::set_last_error("swin_wattn_qkv_proj_prepared_fp8: statistics workspace smaller than "
                         "swin_wattn_qkv_stats_bytes(tokens)");
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  int rc;
  if ((rc = check_device_ptr(x, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(prepared, 256)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(qkv8, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(stats_workspace, 16)) != SWIN_WATTN_OK) return rc;
  if (amax != nullptr && (rc = check_device_ptr(amax, 4)) != SWIN_WATTN_OK) return rc;
  if (status != nullptr && (rc = check_device_ptr(status, 4)) != SWIN_WATTN_OK) return rc;
  const float scales[3] = {scale_q, scale_k, scale_v};
  cudaError_t e = swin::qkv_proj_fp8_launch(x, prepared, qkv8, tokens, C, eps, scales,
                                            reinterpret_cast<unsigned int*>(amax), stats_workspace, status,
                                            reinterpret_cast<cudaStream_t>(stream));
  g_launches += swin::qkv_launches(tokens, C, false);
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_qkv_proj_prepared_fp8");
}

int swin_wattn_proj_residual(const void* o, const void* w_proj, const float* b_proj, const void* residual,
                             void* y, int tokens, int C, int* status, struct CUstream_st* stream) {
  if (tokens < 0) return SWIN_WATTN_ERR_INVALID_ARG;
  if (C < 32 || C > 1536 || C % 32 != 0) return SWIN_WATTN_ERR_UNSUPPORTED;
  if ((int64_t)tokens >= ((int64_t)1 << 31)) return SWIN_WATTN_ERR_UNSUPPORTED;
  if (tokens == 0) return SWIN_WATTN_OK;
  int rc;
  if ((rc = check_device_ptr(o, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(w_proj, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(residual, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(y, 16)) != SWIN_WATTN_OK) return rc;
  if ((rc = check_device_ptr(b_proj, 4)) != SWIN_WATTN_OK) return rc;
  if (status != nullptr && (rc = check_device_ptr(status, 4)) != SWIN_WATTN_OK) return rc;
  const uintptr_t ob = reinterpret_cast<uintptr_t>(o), yb = reinterpret_cast<uintptr_t>(y);
  const uintptr_t bytes = (uintptr_t)tokens * (uintptr_t)C * 2;
  if (ob < yb + bytes && yb < ob + bytes) {
    swin::set_last_error("swin_wattn_proj_residual: y overlaps o");
    return SWIN_WATTN_ERR_INVALID_ARG;
  }
  cudaError_t e = swin::proj_residual_launch(o, w_proj, b_proj, residual, y, tokens, C, status,
                                             reinterpret_cast<cudaStream_t>(stream));
  ++g_launches;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_proj_residual");
}

int swin_wattn_set_fwd_kernel(swin_wattn_plan_t plan, int kernel) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  if (kernel != SWIN_WATTN_KERNEL_AUTO && kernel != SWIN_WATTN_KERNEL_MMA_SYNC &&
      kernel != SWIN_WATTN_KERNEL_TCGEN05)
    return SWIN_WATTN_ERR_INVALID_ARG;
  swin::Plan& p = plan->p;
  const int old = p.fwd_kernel;
  p.fwd_kernel = kernel;
  swin::FwdLaunch L;
  cudaError_t e = swin::fwd_config(p, &L);
  if (e == cudaErrorNotSupported) {
    p.fwd_kernel = old;
    return SWIN_WATTN_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) {
    p.fwd_kernel = old;
    return cuda_fail(e, "swin_wattn_set_fwd_kernel");
  }
  plan->fwd = L;
  return SWIN_WATTN_OK;
}

int swin_wattn_fwd_kernel(swin_wattn_plan_t plan) {
  if (check_plan(plan) != SWIN_WATTN_OK) return -1;
  return plan->fwd.tc ? SWIN_WATTN_KERNEL_TCGEN05 : SWIN_WATTN_KERNEL_MMA_SYNC;
}

int swin_wattn_set_bwd_kernel(swin_wattn_plan_t plan, int kernel) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  if (kernel != SWIN_WATTN_KERNEL_AUTO && kernel != SWIN_WATTN_KERNEL_MMA_SYNC &&
      kernel != SWIN_WATTN_KERNEL_TCGEN05)
    return SWIN_WATTN_ERR_INVALID_ARG;
  swin::Plan& p = plan->p;
  const int old = p.bwd_kernel;
  p.bwd_kernel = kernel;
  swin::BwdLaunch L;
  cudaError_t e = swin::bwd_config(p, &L);
  if (e == cudaErrorNotSupported || (e == cudaSuccess && L.grid == 0 && p.B > 0)) {
    p.bwd_kernel = old;
    return SWIN_WATTN_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) {
    p.bwd_kernel = old;
    return cuda_fail(e, "swin_wattn_set_bwd_kernel");
  }
  plan->bwd = L;
  return SWIN_WATTN_OK;
}

int swin_wattn_bwd_kernel(swin_wattn_plan_t plan) {
  if (check_plan(plan) != SWIN_WATTN_OK) return -1;
  return plan->bwd.tc ? SWIN_WATTN_KERNEL_TCGEN05 : SWIN_WATTN_KERNEL_MMA_SYNC;
}

int swin_wattn_device_status(swin_wattn_plan_t plan, struct CUstream_st* stream) {
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, plan->p.err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && word != 0) e = cudaMemsetAsync(plan->p.err, 0, sizeof(int), st);
  if (e == cudaSuccess && word != 0) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "swin_wattn_device_status");
  if (word != 0) {
    swin::set_last_error("a bounded device wait ran out (tensor-core completion never arrived)");
    return SWIN_WATTN_ERR_TIMEOUT;
  }
  return SWIN_WATTN_OK;
}

int swin_wattn_destroy(swin_wattn_plan_t plan) {
  if (plan == nullptr) return SWIN_WATTN_OK;
  int rc = check_plan(plan);
  if (rc != SWIN_WATTN_OK) return rc;
  {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    g_plans.erase(plan);
  }
  cudaError_t e = cudaDeviceSynchronize();
  plan->p.magic = 0;
  free_pipe(plan->pipe);
  free_plan_buffers(plan->p);
  delete plan;
  return e == cudaSuccess ? SWIN_WATTN_OK : cuda_fail(e, "swin_wattn_destroy");
}

}  // extern "C"
