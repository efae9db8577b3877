// Single-row attention over a KV cache with no memory allocation at all.
//
// Some callers cannot allocate device memory on the path that runs this
// step: code that runs inside a memory-pool budget that is already fully
// handed out, inference servers that forbid allocation after start-up so
// that memory use stays fixed and no call can fail with out-of-memory half
// way through a request, and embedders whose own allocator owns the device.
// For them this file keeps the scratch the split-K attention needs (the
// per-range partial states) in one fixed, file-scope device array instead of
// asking cudaMalloc for it.
//
// Limits and sharing:
//   - the array holds PF_NOALLOC_SCRATCH_FLOATS floats (2 MiB); every GPU
//     that loads this library keeps it until the process exits;
//   - a request needs the tickets of the kernel's last-cluster merge (one
//     int per KV head, rounded up to four) and one folded state per (KV
//     head, cluster of four key ranges): n_kv_head * C * (n_head / n_kv_head
//     * head_dim + 32) floats, C being at most 36 / n_kv_head (at least 1);
//     it is refused (PF_E_ARG) when that is more than the array holds;
//   - every call, on every stream, uses the same array: calls whose work
//     overlaps on the GPU race and give wrong results, so callers must order
//     them (one stream, or events);
//   - the call clears the tickets it uses before its launch; every state it
//     reads is written by the same launch;
//   - its last four floats hold the call's device error word (reset by the
//     call, read back after it).
#include "../../include/prefill_ops.h"
#include "common.cuh"
#include "kernels.h"

#include <mutex>
#include <string>

namespace {

constexpr size_t PF_NOALLOC_SCRATCH_FLOATS = size_t(1) << 19;

// The scratch itself.  In host code this name is only a stand-in for the
// device object; host code must use the address from cudaGetSymbolAddress.
static __device__ __align__(256) float g_noalloc_scratch[PF_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};
int fail(int code, const std::string& m) {
  pf::set_op_error(m);
  return code;
}

// Device address of the scratch array on the current device, looked up on
// the first call made with that device current.
int scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PF_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(PF_E_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(PF_E_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return PF_OK;
}

}  // namespace

extern "C" int pfop_attention_split_noalloc(const void* q_dev, const void* k_dev, const void* v_dev, int32_t Hq,
                                            int32_t Hkv, int32_t hd, int32_t pos, int32_t kv_len, void* out_dev,
                                            void* stream) {
  if (!q_dev || !k_dev || !v_dev || !out_dev || pos < 0 || pos >= kv_len || Hq < 1 || Hkv < 1)
    return fail(PF_E_ARG, "bad argument");
  // the shapes and alignments the kernels take, refused here before any GPU work
  if (hd != 64 && hd != 256) return fail(PF_E_ARG, "head_dim must be 64 or 256");
  if (Hq % Hkv != 0 || Hq / Hkv > 16 || 16 % (Hq / Hkv) != 0)
    return fail(PF_E_ARG, "n_head must be a multiple of n_head_kv with a group size dividing 16");
  if ((reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(k_dev) | reinterpret_cast<uintptr_t>(v_dev)) &
      15)
    return fail(PF_E_ARG, "q, k and v must be 16-byte aligned");
  const size_t need = pf::attn_split_partials_floats(Hq, Hkv, hd, pos);
  if (need > PF_NOALLOC_SCRATCH_FLOATS - 4)
    return fail(PF_E_ARG, "request needs " + std::to_string(need) + " scratch floats; the fixed array holds " +
                              std::to_string(PF_NOALLOC_SCRATCH_FLOATS));
  float* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != PF_OK) return rc;
  pf::AttnArgs a;
  a.q = static_cast<const __half*>(q_dev);
  a.k = static_cast<const __half*>(k_dev);
  a.v = static_cast<const __half*>(v_dev);
  a.out = static_cast<__nv_bfloat16*>(out_dev);
  a.M = 1;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.hd = hd;
  a.pos_base = pos;
  a.kv_len = kv_len;
  int* err_word = reinterpret_cast<int*>(scratch + PF_NOALLOC_SCRATCH_FLOATS - 4);
  a.err = err_word;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(err_word, 0, 16, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, pf::attn_split_ticket_bytes(Hkv), s);
  if (e != cudaSuccess) return fail(PF_E_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(e));
  e = pf::launch_attn_split(a, scratch, s);
  if (e != cudaSuccess) return fail(PF_E_CUDA, std::string("attention launch: ") + cudaGetErrorString(e));
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(PF_E_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
  int h = 0;
  e = cudaMemcpy(&h, err_word, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(PF_E_CUDA, std::string("cudaMemcpy: ") + cudaGetErrorString(e));
  if (h) return fail(PF_E_DEVICE_TIMEOUT, "attention gave up a bounded wait, code " + std::to_string(h));
  return PF_OK;
}
