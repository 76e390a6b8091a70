// attn_bwd_fixed_scratch: the whole dense/THD backward (preprocess, main pass
// with fp32 atomic dQ accumulation, postprocess) for callers that cannot
// allocate device memory.  Delta and the dQ accumulator live in a
// library-owned static device array instead of a caller workspace.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "launch.h"

namespace attn {
namespace {

// 16 MiB of scratch, held by every GPU that loads the library until exit.
static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_FIXED_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  unsigned long long ctx_id;  // context the address was taken in (0: none yet)
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Unique id of the current context (never reused within a process, unlike a
// context handle); 0 when it cannot be read.
unsigned long long current_context_id() {
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  if (!get_id || !get_cur) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_bwd_scratch on the current device.  The host-side name is
// only a stand-in, so the address is looked up with the device current and
// cached together with the id of the context it belongs to; after a device
// reset (a new primary context, the module loaded again) the id differs and the
// address is looked up again.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaFree(nullptr);  // makes the primary context current (no allocation)
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& c = g_scratch[dev];
  if (!c.ptr || ctx == 0 || c.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    c.ptr = p;
    c.ctx_id = ctx;
  }
  *out = c.ptr;
  return cudaSuccess;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" attn_status_t attn_bwd_fixed_scratch(const attn_problem_t* p, const void* q,
                                                const void* k, const void* v, const void* o,
                                                const void* dout, const float* lse, void* dq,
                                                void* dk, void* dv, attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o) ||
      !is_aligned16(dout) || !is_aligned16(lse) || !is_aligned16(dq) || !is_aligned16(dk) ||
      !is_aligned16(dv))
    return ATTN_ERR_ALIGNMENT;
  // Validate before any size is computed from the problem's fields.
  bool empty = false;
  const attn_status_t valid = validate_dense_problem(p, &empty);
  if (valid != ATTN_OK) return valid;
  if (empty) return ATTN_OK;
  const size_t acc_bytes = attn_bwd_workspace_size(p, ATTN_DQ_ATOMIC);
  if (acc_bytes == 0) return ATTN_ERR_INVALID_ARG;
  // scratch layout: [dQ accumulator fp32 rows*Hq*D][Delta fp32 rows*Hq]
  const bool thd = p->cu_seqlens != nullptr;
  const size_t rows = thd ? static_cast<size_t>(p->capacity)
                          : static_cast<size_t>(p->batch) * static_cast<size_t>(p->seqlen);
  const size_t delta_off = (acc_bytes + 255) / 256 * 256;
  const size_t need = delta_off + rows * static_cast<size_t>(p->heads_q) * 4;
  if (need > ATTN_FIXED_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  float* acc = static_cast<float*>(scratch);
  float* delta = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + delta_off);

  // The three stages of the regular backward, run in ATOMIC mode with the
  // accumulator (cleared by the preprocess) and Delta taken from the scratch.
  attn_status_t s = attn_bwd_preprocess(p, ATTN_DQ_ATOMIC, o, dout, delta, acc,
                                        acc_bytes, stream);
  if (s != ATTN_OK) return s;
  s = attn_bwd(p, ATTN_DQ_ATOMIC, q, k, v, dout, lse, delta, dk, dv, acc,
               acc_bytes, stream);
  if (s != ATTN_OK) return s;
  return attn_bwd_postprocess(p, ATTN_DQ_ATOMIC, acc, acc_bytes, dq, dk, dv,
                              stream);
}
