// apa_noalloc.cu -- apa_quantize_noalloc: the NVFP4 quantizer without any
// device allocation.
//
// Some callers cannot allocate device memory on the call path: runtimes that
// hand every byte of the GPU to their own arena at start-up and forbid driver
// allocations afterwards, plugin interfaces that pass buffers in but offer no
// allocator, and latency-critical loops where a cudaMalloc (which may
// synchronize the device) is not acceptable.  For them this entry point keeps
// the quantizer's temporary statistics (per-tile key sums, per-channel key
// min/max, per-head max |v|, |q| and |k - mu|) in one fixed array that lives in the
// library's device image instead of a stream-ordered allocation.  The caller
// still passes every input and output buffer.
#include <mutex>

#include "../../include/apa.h"
#include "apa_internal.h"

namespace apa {

namespace {

// The scratch array.  Every GPU that loads the library holds it until the
// process exits.  In host code this name is only a host-side stand-in for the
// symbol; kernels must be given the device address from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_quant_scratch[APA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
uint8_t* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_quant_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_addr[dev] = static_cast<uint8_t*>(ptr);
  }
  return g_scratch_addr[dev];
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

}  // namespace apa

extern "C" size_t apa_quantize_noalloc_scratch_bytes(int B, int Hq, int Hkv, int Nkv, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nkv < 1 || d < 1) return 0;
  const size_t BH = (size_t)B * Hkv, T = (Nkv + apa::kTile - 1) / apa::kTile, BHq = (size_t)B * Hq;
  return apa::align256(BH * T * d * 4) + 2 * apa::align256(BH * d * 4) + apa::align256(BH * 4) +
         apa::align256(BHq * 4) + apa::align256(BH * 4);
}

extern "C" int apa_quantize_noalloc(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq,
                                    int Nkv, int d, uint8_t* kv_blob, uint8_t* q_blob, float* mu, float* s_q,
                                    float* s_k, float* s_v, cudaStream_t stream) {
  if (!q || !k || !v || !kv_blob || !q_blob || !mu || !s_q || !s_k || !s_v) return APA_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || Hq % Hkv) return APA_ERR_SHAPE;
  if ((Nkv + apa::kTile - 1) / apa::kTile > 65535) return APA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return APA_ERR_HEAD_DIM;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v) & 15) return APA_ERR_ALIGN;
  const size_t need = apa_quantize_noalloc_scratch_bytes(B, Hq, Hkv, Nkv, d);
  if (need > (size_t)APA_NOALLOC_SCRATCH_BYTES) return APA_ERR_SCRATCH;
  uint8_t* scratch = apa::scratch_address();
  if (!scratch) return APA_ERR_CUDA;
  apa::Shape s{B, Hq, Hkv, Nq, Nkv, d, 0};
  const size_t BH = s.BH(), T = s.T(), BHq = (size_t)B * Hq;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = scratch + off;
    off += apa::align256(bytes);
    return p;
  };
  apa::Workspace ws{};
  ws.ksum = (float*)take(BH * T * d * 4);
  ws.kmin = (uint32_t*)take(BH * d * 4);
  ws.kmax = (uint32_t*)take(BH * d * 4);
  ws.vamax = (uint32_t*)take(BH * 4);
  ws.qamax = (uint32_t*)take(BHq * 4);
  ws.kcamax = (uint32_t*)take(BH * 4);
  ws.mu = mu;
  ws.s_k = s_k;
  ws.s_v = s_v;
  ws.s_q = s_q;
  ws.kv_blob = kv_blob;
  ws.q_blob = q_blob;
  // launch_quantize resets the min / max words (the array keeps the previous
  // call's contents) and overwrites every per-tile sum before reading it.
  return apa::launch_quantize(s, q, k, v, ws, true, true, stream) == cudaSuccess ? APA_OK : APA_ERR_CUDA;
}
