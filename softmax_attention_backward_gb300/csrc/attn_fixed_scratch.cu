// attn_bwd_fixed_scratch: the whole dense/THD backward (preprocess, main pass
// with fp32 atomic dQ accumulation, postprocess) for callers that cannot
// allocate device memory.  Delta and the dQ accumulator live in a
// library-owned static device array instead of a caller workspace.
#include <cuda_runtime.h>

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
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device.  The host-side name is
// only a stand-in, so the address is looked up once per device (with that
// device current) and cached.
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  if (p->heads_q <= 0 || p->heads_kv <= 0 || p->heads_q % p->heads_kv || !std::isfinite(p->scale))
    return ATTN_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(o) ||
      !is_aligned16(dout) || !is_aligned16(lse) || !is_aligned16(dq) || !is_aligned16(dk) ||
      !is_aligned16(dv))
    return ATTN_ERR_ALIGNMENT;
  const bool thd = p->cu_seqlens != nullptr;
  const int64_t rows = thd ? p->capacity : static_cast<int64_t>(p->batch) * p->seqlen;
  if (rows < 0) return ATTN_ERR_INVALID_ARG;
  if (rows == 0) return ATTN_OK;
  // scratch layout: [dQ accumulator fp32 rows*Hq*D][Delta fp32 rows*Hq]
  const int64_t acc_bytes = rows * p->heads_q * p->head_dim * 4;
  const int64_t delta_off = (acc_bytes + 255) / 256 * 256;
  const int64_t need = delta_off + rows * p->heads_q * 4;
  if (need > ATTN_FIXED_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;

  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return ATTN_ERR_CUDA;
  float* acc = static_cast<float*>(scratch);
  float* delta = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + delta_off);

  // The three stages of the regular backward, run in ATOMIC mode with the
  // accumulator (cleared by the preprocess) and Delta taken from the scratch.
  attn_status_t s = attn_bwd_preprocess(p, ATTN_DQ_ATOMIC, o, dout, delta, acc,
                                        static_cast<size_t>(acc_bytes), stream);
  if (s != ATTN_OK) return s;
  s = attn_bwd(p, ATTN_DQ_ATOMIC, q, k, v, dout, lse, delta, dk, dv, acc,
               static_cast<size_t>(acc_bytes), stream);
  if (s != ATTN_OK) return s;
  return attn_bwd_postprocess(p, ATTN_DQ_ATOMIC, acc, static_cast<size_t>(acc_bytes), dq, dk, dv,
                              stream);
}
