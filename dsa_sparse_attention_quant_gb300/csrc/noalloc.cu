// noalloc.cu — dsa_indexer_logits_topk_static: the fused indexer call for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a scratch buffer:
// plugins that only receive the tensors of an op (inputs and outputs, no
// allocator), code whose device memory belongs to a framework allocator it may
// not call, and latency-critical loops that must not touch the allocator. For them this
// entry point takes its scratch from one statically sized device array that
// belongs to the library: every GPU that loads the library holds
// kStaticWorkspaceBytes of device memory for it until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents. Each call's first kernel (the prologue) writes the plan and clears
// the score histograms and top-k counters before the later kernels read them.
// Calls whose kernels overlap on the GPU (two streams, or two host threads)
// race on the array; serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dsaidx.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t{DSA_STATIC_WORKSPACE_BYTES};
constexpr int kMaxDevices = 64;

// Device scratch of the static entry point. In host code this name is only a
// host-side handle; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_static_mutex;
void* g_static_addr[kMaxDevices];                  // device address of the array, per device
unsigned long long g_static_ctx[kMaxDevices];      // id of the context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The process-unique id of the current context (the driver never reuses one),
// or false when there is none yet. Called under g_static_mutex.
bool current_context_id(unsigned long long* id) {
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) != cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || a == nullptr ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
        qb != cudaDriverEntryPointSuccess || b == nullptr)
      return false;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// The device address of the array in the current device's context. It is
// looked up (cudaGetSymbolAddress, with that device current) on the first
// call on a device, and again whenever the device's context has changed since
// (after cudaDeviceReset the array lives at a new address in a new context).
int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ENODEV;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  if (g_static_addr[dev] == nullptr || !have_ctx || g_static_ctx[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return e == cudaErrorNoKernelImageForDevice ? DSA_ENODEV : DSA_ECUDA;
    }
    // the lookup made the device's context current if it was not yet
    if (!current_context_id(&ctx)) return DSA_ECUDA;
    g_static_addr[dev] = p;
    g_static_ctx[dev] = ctx;
  }
  *out = g_static_addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_indexer_logits_topk_static(const DsaBatch* batch, const uint8_t* q_fp8, const float* w_folded,
                                   uint8_t* k_cache, int32_t topk, int32_t* topk_out, const void* k_new,
                                   const int64_t* slot_mapping, int32_t* dev_err, dsa_stream_t stream) {
  const size_t need = dsa_indexer_workspace_size(batch, topk);
  if (need == 0) return DSA_EINVAL;
  if (need > kStaticWorkspaceBytes) return DSA_ENOSPACE;
  if (batch->num_tokens == 0) return DSA_OK;
  void* ws = nullptr;
  const int st = static_workspace(&ws);
  if (st != DSA_OK) return st;
  return dsa_indexer_logits_topk(batch, q_fp8, w_folded, k_cache, topk, topk_out, ws, kStaticWorkspaceBytes, k_new,
                                 slot_mapping, dev_err, stream);
}

}  // extern "C"
