// apa.cu -- the C ABI: argument checks, workspace layout and the launch
// sequence stats -> finalize -> quantize -> pass 1 -> pass 2 (+ merge).
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/apa.h"
#include "apa_internal.h"

#ifndef APA_HOST_LANE_PRIORITY
#define APA_HOST_LANE_PRIORITY 1  // later compute lanes of apa_attention_host at higher stream priority
#endif
#ifndef APA_HOST_WIDE_EIGHTHS
#define APA_HOST_WIDE_EIGHTHS 2  // eighths of the sub-problems of apa_attention_host run in the wide form
#endif

namespace apa {

namespace {

__device__ int g_device_error;  // set by bounded waits that gave up

constexpr size_t kAlign = 256;
constexpr unsigned kKnownFlags =
    APA_FLAG_Q_RESIDUAL | APA_FLAG_LSE_SCALES | APA_FLAG_VALUE_WEIGHTED | APA_FLAG_ROWSUM_MMA;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

__global__ void visible_mask_kernel(Shape s, uint32_t* mask) {
  const int ngroups = s.ngroups(), T = s.T(), nwords = (T + 31) / 32;
  const size_t total = (size_t)s.BH() * ngroups * nwords;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int w = (int)(i % nwords);
    const int grp = (int)((i / nwords) % ngroups);
    const int last_row = min(s.R(), (grp + 1) * kGroupRows) - 1;
    const int t_last = s.causal ? min(T - 1, (last_row / s.G() + s.off()) / kTile) : T - 1;
    const int lo = w * 32, hi = min(t_last, lo + 31);
    uint32_t bits = 0;
    if (hi >= lo) bits = (hi - lo == 31) ? 0xFFFFFFFFu : ((1u << (hi - lo + 1)) - 1u);
    mask[i] = bits;
  }
}

int validate(const void* q, const void* k, const void* v, const float* out, int B, int Hq, int Hkv, int Nq, int Nkv,
             int d, int causal, float eps, bool need_out) {
  if (!q || !k || !v || (need_out && !out)) return APA_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || Hq % Hkv) return APA_ERR_SHAPE;
  if (causal && Nkv < Nq) return APA_ERR_SHAPE;
  if ((Nkv + kTile - 1) / kTile > 65535) return APA_ERR_SHAPE;  // tile index is stored in 16 bits
  if ((long long)(Hq / Hkv) * Nq > (1ll << 30)) return APA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return APA_ERR_HEAD_DIM;
  if (std::isnan(eps) || eps < 0.f) return APA_ERR_EPS;
  if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v) & 15) return APA_ERR_ALIGN;
  return APA_OK;
}

}  // namespace

// Per-device staging of the host-buffer entry point.
constexpr int kHostLanes = 8;  // compute streams of the host-buffer entry point
struct HostStaging {
  std::mutex mu;
  uint8_t* buf = nullptr;
  size_t cap = 0;
  bool ready = false;
  cudaStream_t copy = nullptr, lane[kHostLanes] = {};
  cudaEvent_t fork = nullptr, arrived = nullptr, join[kHostLanes] = {};
  uint8_t* reserve(size_t bytes);  // buffer of at least `bytes`, or null
  bool streams_ready();
};
HostStaging& host_staging();

// Device staging for apa_attention_host: one buffer per device, grown on demand
// and kept for the process (cudaMalloc once instead of a stream-ordered
// allocation that the pool hands back to the driver at every synchronize), a
// copy stream, kHostLanes compute streams and their events.
HostStaging& host_staging() {
  static HostStaging hs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  return hs[dev];
}
uint8_t* HostStaging::reserve(size_t bytes) {
  if (bytes <= cap) return buf;
  if (buf) cudaFree(buf);  // synchronizes; the previous call has completed anyway
  buf = nullptr;
  cap = 0;
  if (cudaMalloc((void**)&buf, bytes) != cudaSuccess) {
    buf = nullptr;
    return nullptr;
  }
  cap = bytes;
  return buf;
}
bool HostStaging::streams_ready() {
  if (ready) return true;
  if (cudaStreamCreateWithFlags(&copy, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&arrived, cudaEventDisableTiming) != cudaSuccess)
    return false;
  // Later lanes take later sub-problems, which arrive last and so set the end of the
  // call: their thread blocks go first whenever the GPU's SMs are all taken.
  int least = 0, greatest = 0;
  if (!APA_HOST_LANE_PRIORITY || cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess)
    least = greatest = 0;
  for (int i = 0; i < kHostLanes; ++i) {
    const int prio = least + (greatest - least) * i / (kHostLanes - 1);
    if (cudaStreamCreateWithPriority(&lane[i], cudaStreamNonBlocking, prio) != cudaSuccess ||
        cudaEventCreateWithFlags(&join[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  }
  ready = true;
  return true;
}

int* device_error_word() {
  static int* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

size_t workspace_layout(const Shape& s, bool apa_mode, Workspace* ws, void* base, unsigned flags) {
  Workspace w{};
  const size_t BH = s.BH(), T = s.T(), d = s.d, nblk = s.nblk(), BHq = (size_t)s.B * s.Hq;
  size_t off = 0;
  uint8_t* b = static_cast<uint8_t*>(base);
  auto take = [&](size_t bytes) -> void* {
    void* p = b ? b + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  if (!apa_mode) {  // the all-exact path: the FP16 copy of V for its P.V product
    w.vamax = (uint32_t*)take(BH * 4);
    w.v16 = (uint16_t*)take(BH * s.Nkv * d * 2);
    if (exact_split(s) > 1) {  // the parts of its split walks
      const size_t parts = BH * nblk * exact_split(s) * kBlockRows;
      w.part_o = (float*)take(parts * d * 4);
      w.part_ml = (float2*)take(parts * 8);
    }
    if (ws) *ws = w;
    return off;
  }
  w.ksum = (float*)take(BH * T * d * 4);
  w.kmin = (uint32_t*)take(BH * d * 4);
  w.kmax = (uint32_t*)take(BH * d * 4);
  w.vamax = (uint32_t*)take(BH * 4);
  w.qamax = (uint32_t*)take(BHq * 4);
  w.kcamax = (uint32_t*)take(BH * 4);
  w.mu = (float*)take(BH * d * 4);
  w.s_k = (float*)take(BH * 4);
  w.s_v = (float*)take(BH * 4);
  w.s_q = (float*)take(BHq * 4);
  w.kv_blob = (uint8_t*)take(BH * T * blob_bytes((int)d));
  w.q_blob = (uint8_t*)take(BH * nblk * qblob_bytes((int)d));
  w.state_o = (float*)take(BH * nblk * kBlockRows * d * 4);
  w.state_ml = (float2*)take(BH * nblk * kBlockRows * 8);
  w.hot_list = (uint32_t*)take(BH * nblk * T * 4);
  w.hot_count = (uint32_t*)take(BH * nblk * 4);
  w.p2_order = (uint32_t*)take(BH * nblk * 4);
  if (flags & APA_FLAG_Q_RESIDUAL) w.q2_blob = (uint8_t*)take(BH * nblk * qblob_bytes((int)d));
  w.kv_ready = (uint32_t*)take((BH * T + 1) * 4);
  if (flags & APA_FLAG_VALUE_WEIGHTED) {
    w.wv = (float*)take(BH * T * 4);
    w.vtsum = (float*)take(BH * T * 4);
  }
  w.v16 = (uint16_t*)take(BH * s.Nkv * d * 2);
  if (apa_split(s) > 1) {  // the parts of pass 2's split walks
    const size_t parts = BH * nblk * apa_split(s) * kBlockRows;
    w.part_o = (float*)take(parts * d * 4);
    w.part_ml = (float2*)take(parts * 8);
    w.part_qmu = (float*)take(BH * nblk * kBlockRows * 4);
  }
  if (ws) *ws = w;
  return off;
}

cudaError_t launch_visible_mask(const Shape& s, uint32_t* hot_mask, cudaStream_t st) {
  visible_mask_kernel<<<256, 256, 0, st>>>(s, hot_mask);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ stage timing
// Opt-in measurement aid: events recorded on the call's stream before the
// quantizer, before pass 1, before pass 2 and after pass 2.
namespace {
struct StageTiming {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> ev;  // 4 per recorded call
  size_t used = 0;
} g_timing;

size_t begin_call() {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  if (!g_timing.on) return SIZE_MAX;
  if (g_timing.used * 4 + 4 > g_timing.ev.size()) {
    for (int i = 0; i < 4; ++i) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return SIZE_MAX;
      g_timing.ev.push_back(e);
    }
  }
  return g_timing.used++;
}
}  // namespace

static int run_attention(const Shape& s, const void* q, const void* k, const void* v, float eps, float* out, float* lse,
                         uint32_t* hot_mask, void* workspace, cudaStream_t stream, bool wide_pass1 = false,
                         unsigned flags = 0, bool kv_in_pass1_ok = true) {
  const size_t call = begin_call();
  auto stage = [&](int slot) {
    if (call != SIZE_MAX) cudaEventRecord(g_timing.ev[call * 4 + slot], stream);
  };
  Workspace ws;
  if (eps == 0.f) {
    // all exact: the FP16 copy of V, then pass 2 over every visible tile
    workspace_layout(s, false, &ws, workspace, flags);
    stage(0);
    if (launch_v16(s, v, ws, stream) != cudaSuccess) return APA_ERR_CUDA;
    stage(1);
    if (hot_mask && launch_visible_mask(s, hot_mask, stream) != cudaSuccess) return APA_ERR_CUDA;
    stage(2);
    const int st = launch_pass2(s, q, k, v, &ws, out, lse, stream) == cudaSuccess ? APA_OK : APA_ERR_CUDA;
    stage(3);
    return st;
  }
  workspace_layout(s, true, &ws, workspace, flags);
  stage(0);
  if (hot_mask) {
    const size_t words = (size_t)s.BH() * s.ngroups() * ((s.T() + 31) / 32);
    if (cudaMemsetAsync(hot_mask, 0, words * 4, stream) != cudaSuccess) return APA_ERR_CUDA;
  }
  // The K/V tiles are quantized inside the pass-1 launch, on the SMs its CTAs
  // leave free, when there are enough of those; the statistics and Q come first.
  // The least-squared-error scales cost about three times the quantizer work, more
  // than those SMs keep up with, so that option keeps the quantizer kernel.
  const bool lse_scales = (flags & APA_FLAG_LSE_SCALES) != 0, wide = wide_pass1 || ws.q2_blob;
  const bool rowsum_mma = (flags & APA_FLAG_ROWSUM_MMA) != 0;
  const bool kv_in_pass1 =
      kv_in_pass1_ok && !lse_scales && pass1_quantizes_kv(s, wide_pass1, ws.q2_blob != nullptr, rowsum_mma);
  if (launch_quantize(s, q, k, v, ws, true, true, stream, lse_scales, kv_in_pass1) != cudaSuccess)
    return APA_ERR_CUDA;
  stage(1);
  const KvSource src{k, v, lse_scales};
  cudaError_t e1 = launch_pass1(s, ws, eps, hot_mask, wide, stream, kv_in_pass1 ? &src : nullptr, rowsum_mma);
  if (kv_in_pass1 && e1 == cudaErrorCooperativeLaunchTooLarge) {
    // fewer SMs than the device reports are ours (a partitioned or shared GPU):
    // quantize K/V with the separate kernel (recomputing the same statistics) and
    // run pass 1 on its own
    (void)cudaGetLastError();
    if (launch_quantize(s, q, k, v, ws, false, true, stream, lse_scales) != cudaSuccess) return APA_ERR_CUDA;
    e1 = launch_pass1(s, ws, eps, hot_mask, wide, stream, nullptr, rowsum_mma);
  }
  if (e1 != cudaSuccess) return APA_ERR_CUDA;
  if (launch_pass2_order(s, ws, stream) != cudaSuccess) return APA_ERR_CUDA;
  stage(2);
  if (launch_pass2(s, q, k, v, &ws, out, lse, stream) != cudaSuccess) return APA_ERR_CUDA;
  stage(3);
  return APA_OK;
}

}  // namespace apa

using apa::Shape;

extern "C" {

size_t apa_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || Hq % Hkv) return 0;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, 1};
  return apa::workspace_layout(s, eps != 0.f, nullptr, nullptr);
}

int apa_attention_ws(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                     int causal, float eps, float* out, float* lse, uint32_t* hot_mask, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  int st = apa::validate(q, k, v, out, B, Hq, Hkv, Nq, Nkv, d, causal, eps, true);
  if (st) return st;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, causal ? 1 : 0};
  const size_t need = apa::workspace_layout(s, eps != 0.f, nullptr, nullptr);
  if (need > 0 && (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255))) return APA_ERR_NOMEM;
  return apa::run_attention(s, q, k, v, eps, out, lse, hot_mask, workspace, stream);
}

int apa_attention(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                  int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream) {
  int st = apa::validate(q, k, v, out, B, Hq, Hkv, Nq, Nkv, d, causal, eps, true);
  if (st) return st;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, causal ? 1 : 0};
  const size_t need = apa::workspace_layout(s, eps != 0.f, nullptr, nullptr);
  void* ws = nullptr;
  if (need && cudaMallocAsync(&ws, need, stream) != cudaSuccess) return APA_ERR_NOMEM;
  st = apa::run_attention(s, q, k, v, eps, out, lse, hot_mask, ws, stream);
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess && st == APA_OK) st = APA_ERR_CUDA;
  return st;
}

int apa_attention_paged(const void* q, const void* k_pages, const void* v_pages, int num_pages,
                        const int32_t* block_table, int max_pages, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                        int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream) {
  int st = apa::validate(q, k_pages, v_pages, out, B, Hq, Hkv, Nq, Nkv, d, causal, eps, true);
  if (st) return st;
  if (!block_table) return APA_ERR_NULL;
  if (num_pages < 1 || max_pages < (Nkv + apa::kTile - 1) / apa::kTile ||
      (long long)num_pages * Hkv * apa::kTile > (1ll << 31))
    return APA_ERR_SHAPE;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, causal ? 1 : 0};
  s.pages = block_table;
  s.max_pages = max_pages;
  s.num_pages = num_pages;
  const size_t need = apa::workspace_layout(s, eps != 0.f, nullptr, nullptr);
  void* ws = nullptr;
  if (need && cudaMallocAsync(&ws, need, stream) != cudaSuccess) return APA_ERR_NOMEM;
  st = apa::run_attention(s, q, k_pages, v_pages, eps, out, lse, hot_mask, ws, stream);
  if (ws && cudaFreeAsync(ws, stream) != cudaSuccess && st == APA_OK) st = APA_ERR_CUDA;
  return st;
}

size_t apa_workspace_bytes_ex(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps, unsigned flags) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || Hq % Hkv || (flags & ~apa::kKnownFlags)) return 0;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, 1};
  return apa::workspace_layout(s, eps != 0.f, nullptr, nullptr, flags);
}

int apa_attention_ex(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                     int causal, float eps, unsigned flags, float* out, float* lse, uint32_t* hot_mask,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  int st = apa::validate(q, k, v, out, B, Hq, Hkv, Nq, Nkv, d, causal, eps, true);
  if (st) return st;
  if (flags & ~apa::kKnownFlags) return APA_ERR_FLAGS;
  // the ones-MMA row sums and the residual Q term both need the same TMEM columns
  if ((flags & APA_FLAG_ROWSUM_MMA) && (flags & APA_FLAG_Q_RESIDUAL)) return APA_ERR_FLAGS;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, causal ? 1 : 0};
  const size_t need = apa::workspace_layout(s, eps != 0.f, nullptr, nullptr, flags);
  void* ws = workspace;
  if (ws && (workspace_bytes < need || ((uintptr_t)ws & 255))) return APA_ERR_NOMEM;  // as apa_attention_ws
  if (!ws && need && cudaMallocAsync(&ws, need, stream) != cudaSuccess) return APA_ERR_NOMEM;
  st = apa::run_attention(s, q, k, v, eps, out, lse, hot_mask, ws, stream, false, flags);
  if (!workspace && ws && cudaFreeAsync(ws, stream) != cudaSuccess && st == APA_OK) st = APA_ERR_CUDA;
  return st;
}

int apa_attention_host(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                       int causal, float eps, float* out, float* lse, uint32_t* hot_mask, cudaStream_t stream) {
  int st = apa::validate(q, k, v, out, B, Hq, Hkv, Nq, Nkv, d, causal, eps, true);
  if (st) return st;
  // Each (b, KV head) is a problem of its own for the method (per-head scales and
  // key mean, its own query heads and keys), so the call runs as BH sub-problems
  // B = 1, Hq = G, Hkv = 1: the inputs of one travel on the copy stream while
  // earlier ones compute on up to kHostLanes streams, and each one's results go
  // back as soon as it is done.  The results are those of one apa_attention call.
  const int G = Hq / Hkv, BH = B * Hkv;
  const Shape sub{1, G, 1, Nq, Nkv, d, causal ? 1 : 0};
  const size_t qh = (size_t)G * Nq * d, kh = (size_t)Nkv * d, lh = (size_t)G * Nq;
  const size_t mh = (size_t)sub.ngroups() * ((sub.T() + 31) / 32);
  const size_t need = apa::workspace_layout(sub, eps != 0.f, nullptr, nullptr);
  const int L = BH < apa::kHostLanes ? BH : apa::kHostLanes;
  // The last sub-problems to arrive finish sooner with one block per pass-1 CTA,
  // spread over the SMs the earlier ones leave free; with the lanes' stream
  // priorities the last 2/8 was the best split measured on the 8-head
  // 2048 x 122880 layer (4.73 ms, against 5.0 for 3/8 and 5.15 for none).
  const int wide_from = BH - (APA_HOST_WIDE_EIGHTHS * BH) / 8;
  size_t off = 0;
  auto slot = [&](size_t bytes) {
    const size_t o = off;
    off += apa::align_up(bytes);
    return o;
  };
  const size_t oq = slot(BH * qh * 2), ok = slot(BH * kh * 2), ov = slot(BH * kh * 2), oo = slot(BH * qh * 4);
  const size_t ol = slot(lse ? BH * lh * 4 : 0), om = slot(hot_mask ? BH * mh * 4 : 0);
  const size_t ow = slot(L * apa::align_up(need));
  // one call at a time per device: the device buffer and the streams are the library's
  apa::HostStaging& hs = apa::host_staging();
  std::lock_guard<std::mutex> lk(hs.mu);
  uint8_t* dev = hs.reserve(off);
  if (!dev) return APA_ERR_NOMEM;
  if (!hs.streams_ready()) return APA_ERR_CUDA;
  auto ok_ = [](cudaError_t e) { return e == cudaSuccess; };
  bool good = ok_(cudaEventRecord(hs.fork, stream)) && ok_(cudaStreamWaitEvent(hs.copy, hs.fork, 0));
  for (int i = 0; i < L && good; ++i) good = ok_(cudaStreamWaitEvent(hs.lane[i], hs.fork, 0));
  st = good ? APA_OK : APA_ERR_CUDA;
  for (int j = 0; j < BH && st == APA_OK; ++j) {
    cudaStream_t ls = hs.lane[j % L];
    uint8_t *dq = dev + oq + j * qh * 2, *dk = dev + ok + j * kh * 2, *dv = dev + ov + j * kh * 2;
    float* dout = (float*)(dev + oo) + j * qh;
    float* dlse = lse ? (float*)(dev + ol) + j * lh : nullptr;
    uint32_t* dmask = hot_mask ? (uint32_t*)(dev + om) + j * mh : nullptr;
    good = ok_(cudaMemcpyAsync(dq, (const uint16_t*)q + j * qh, qh * 2, cudaMemcpyHostToDevice, hs.copy)) &&
           ok_(cudaMemcpyAsync(dk, (const uint16_t*)k + j * kh, kh * 2, cudaMemcpyHostToDevice, hs.copy)) &&
           ok_(cudaMemcpyAsync(dv, (const uint16_t*)v + j * kh, kh * 2, cudaMemcpyHostToDevice, hs.copy)) &&
           ok_(cudaEventRecord(hs.arrived, hs.copy)) && ok_(cudaStreamWaitEvent(ls, hs.arrived, 0));
    if (!good) {
      st = APA_ERR_CUDA;
      break;
    }
    st = apa::run_attention(sub, dq, dk, dv, eps, dout, dlse, dmask,
                            need ? dev + ow + (j % L) * apa::align_up(need) : nullptr, ls, j >= wide_from, 0,
                            false);  // (sub-problems share the GPU: no whole-GPU cooperative launch)
    if (st != APA_OK) break;
    good = ok_(cudaMemcpyAsync(out + j * qh, dout, qh * 4, cudaMemcpyDeviceToHost, ls)) &&
           (!lse || ok_(cudaMemcpyAsync(lse + j * lh, dlse, lh * 4, cudaMemcpyDeviceToHost, ls))) &&
           (!hot_mask || ok_(cudaMemcpyAsync(hot_mask + j * mh, dmask, mh * 4, cudaMemcpyDeviceToHost, ls)));
    if (!good) st = APA_ERR_CUDA;
  }
  // join every lane into `stream` (also after an error, so nothing is left in flight)
  for (int i = 0; i < L; ++i)
    if (!ok_(cudaEventRecord(hs.join[i], hs.lane[i])) || !ok_(cudaStreamWaitEvent(stream, hs.join[i], 0)))
      if (st == APA_OK) st = APA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess && st == APA_OK) st = APA_ERR_CUDA;
  return st;
}

int apa_workspace_operands(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float eps, unsigned flags,
                           size_t* kv_blob, size_t* q_blob, size_t* mu, size_t* s_q, size_t* s_k, size_t* s_v) {
  if (!kv_blob || !q_blob || !mu || !s_q || !s_k || !s_v) return APA_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || Hq % Hkv) return APA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return APA_ERR_HEAD_DIM;
  if (std::isnan(eps) || eps <= 0.f) return APA_ERR_EPS;  // the all-exact path quantizes nothing
  if (flags & ~apa::kKnownFlags) return APA_ERR_FLAGS;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, 1};
  apa::Workspace w;
  apa::workspace_layout(s, true, &w, reinterpret_cast<void*>(uintptr_t(4096)), flags);
  auto off = [](const void* p) { return (size_t)(reinterpret_cast<uintptr_t>(p) - 4096); };
  *kv_blob = off(w.kv_blob);
  *q_blob = off(w.q_blob);
  *mu = off(w.mu);
  *s_q = off(w.s_q);
  *s_k = off(w.s_k);
  *s_v = off(w.s_v);
  return APA_OK;
}

size_t apa_kv_blob_bytes(int B, int Hkv, int Nkv, int d) {
  if (B < 1 || Hkv < 1 || Nkv < 1) return 0;
  return (size_t)B * Hkv * ((Nkv + apa::kTile - 1) / apa::kTile) * apa::blob_bytes(d);
}

size_t apa_q_blob_bytes(int B, int Hq, int Hkv, int Nq, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Hq % Hkv) return 0;
  Shape s{B, Hq, Hkv, Nq, 1, d, 0};
  return (size_t)s.BH() * s.nblk() * apa::qblob_bytes(d);
}

int apa_quantize(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                 uint8_t* kv_blob, uint8_t* q_blob, float* mu, float* s_q, float* s_k, float* s_v,
                 cudaStream_t stream) {
  return apa_quantize_ex(q, k, v, B, Hq, Hkv, Nq, Nkv, d, 0u, kv_blob, q_blob, nullptr, mu, s_q, s_k, s_v, stream);
}

int apa_quantize_ex(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                    unsigned flags, uint8_t* kv_blob, uint8_t* q_blob, uint8_t* q2_blob, float* mu, float* s_q,
                    float* s_k, float* s_v, cudaStream_t stream) {
  int st = apa::validate(q, k, v, nullptr, B, Hq, Hkv, Nq, Nkv, d, 0, 1.f, false);
  if (st) return st;
  if (!kv_blob || !q_blob || !mu || !s_q || !s_k || !s_v) return APA_ERR_NULL;
  if (flags & ~apa::kKnownFlags) return APA_ERR_FLAGS;
  Shape s{B, Hq, Hkv, Nq, Nkv, d, 0};
  const size_t BH = s.BH(), T = s.T(), BHq = (size_t)B * Hq;
  // scratch: per-tile key sums and the min / max / amax words
  size_t off = 0;
  auto slot = [&](size_t bytes) {
    const size_t o = off;
    off += apa::align_up(bytes);
    return o;
  };
  const size_t o_sum = slot(BH * T * d * 4), o_min = slot(BH * d * 4), o_max = slot(BH * d * 4), o_va = slot(BH * 4),
               o_qa = slot(BHq * 4), o_kc = slot(BH * 4);
  uint8_t* scratch = nullptr;
  if (cudaMallocAsync((void**)&scratch, off, stream) != cudaSuccess) return APA_ERR_NOMEM;
  apa::Workspace ws{};
  ws.ksum = (float*)(scratch + o_sum);
  ws.kmin = (uint32_t*)(scratch + o_min);
  ws.kmax = (uint32_t*)(scratch + o_max);
  ws.vamax = (uint32_t*)(scratch + o_va);
  ws.qamax = (uint32_t*)(scratch + o_qa);
  ws.kcamax = (uint32_t*)(scratch + o_kc);
  ws.mu = mu;
  ws.s_k = s_k;
  ws.s_v = s_v;
  ws.s_q = s_q;
  ws.kv_blob = kv_blob;
  ws.q_blob = q_blob;
  ws.q2_blob = q2_blob;
  st = apa::launch_quantize(s, q, k, v, ws, true, true, stream, (flags & APA_FLAG_LSE_SCALES) != 0) == cudaSuccess
           ? APA_OK
           : APA_ERR_CUDA;
  if (cudaFreeAsync(scratch, stream) != cudaSuccess && st == APA_OK) st = APA_ERR_CUDA;
  return st;
}

int apa_stage_timing(int enable) {
  std::lock_guard<std::mutex> lk(apa::g_timing.mu);
  apa::g_timing.on = enable != 0;
  apa::g_timing.used = 0;
  return APA_OK;
}

int apa_stage_timing_read(float* ms, int* calls) {
  if (!ms || !calls) return APA_ERR_NULL;
  std::lock_guard<std::mutex> lk(apa::g_timing.mu);
  for (int i = 0; i < 3; ++i) ms[i] = 0.f;
  for (size_t c = 0; c < apa::g_timing.used; ++c) {
    if (cudaEventSynchronize(apa::g_timing.ev[c * 4 + 3]) != cudaSuccess) return APA_ERR_CUDA;
    for (int i = 0; i < 3; ++i) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, apa::g_timing.ev[c * 4 + i], apa::g_timing.ev[c * 4 + i + 1]) != cudaSuccess)
        return APA_ERR_CUDA;
      ms[i] += t;
    }
  }
  *calls = (int)apa::g_timing.used;
  apa::g_timing.used = 0;
  return APA_OK;
}

int apa_check_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return APA_ERR_CUDA;
  int* w = apa::device_error_word();
  if (!w) return APA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return APA_ERR_CUDA;
  if (h) {
    const int zero = 0;
    cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return APA_ERR_DEVICE;
  }
  return APA_OK;
}

const char* apa_status_string(int status) {
  switch (status) {
    case APA_OK: return "ok";
    case APA_ERR_NULL: return "a required pointer is null";
    case APA_ERR_SHAPE: return "invalid shape (B, Hq, Hkv, Nq, Nkv; Hq % Hkv; causal needs Nkv >= Nq)";
    case APA_ERR_EPS: return "eps must be >= 0 and not NaN (> 0 where pass-1 operands are asked for)";
    case APA_ERR_HEAD_DIM: return "head dimension must be 64, 128 or 256";
    case APA_ERR_CUDA: return "CUDA error (see cudaGetLastError)";
    case APA_ERR_NOMEM: return "workspace allocation failed or workspace too small";
    case APA_ERR_DEVICE: return "a kernel recorded a device-side error (a wait timed out, or a block-table entry was outside the page pool)";
    case APA_ERR_ALIGN: return "q, k and v must be 16-byte aligned";
    case APA_ERR_SCRATCH: return "problem too large for the fixed scratch of apa_quantize_noalloc";
    case APA_ERR_FLAGS: return "unknown option flag";
  }
  return "unknown status";
}

}  // extern "C"
