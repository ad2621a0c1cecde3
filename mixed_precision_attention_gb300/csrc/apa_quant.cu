// apa_quant.cu -- per-head statistics and the NVFP4 quantizer.
//
// "APA: sloppy attention, exact where it counts" (rfriedmann.de blog),
// section "Pass 1: FP4 everywhere, with a hot test": operands are E2M1 with one
// UE4M3 scale per 16 values and one FP32 scale per head, so the head's largest
// magnitude maps to 6 * 448 = 2688; keys are mean-centred per channel first
// ("Mean-centred K"), and a prep stage writes K and V^T as one blob per 64-key
// tile ("A 9216-byte blob per tile").
//
// The quantizer is bit-exact by construction: every FP32 operation is an
// explicitly rounded intrinsic (no contraction), in this order per 16-block:
//   a = max|x|;  sb = UE4M3_rn_sat(a / (6 s));  if sb == 0 all codes are 0,
//   else code = E2M1_rn_sat(x * rcp_rn(UE4M3(sb) * s)).
// The key mean is an FP32 sum per 64-key tile in ascending key order; the tile
// sums are added in FP64 per range of 64 consecutive tiles (ascending), the
// range sums in ascending order; divided by Nkv in FP64 and rounded to FP32.
//
// Kernels:
//   stats_kernel     K/V tiles (bulk-copied to shared memory): per-tile FP32 key
//                    sums, per-channel min/max of K (atomics on an order-preserving
//                    encoding: exact, so order-free), max |V|; Q rows: max |Q| per
//                    query head.
//                    With the value-weighted hot test also each key's value norm
//                    and per tile their maximum and FP32 sum.
//   finalize_kernel  per (b, KV head, 8 channels): mu and the head's max |k - mu|;
//                    per (b, KV head), value-weighted: the mean key value norm and
//                    the tiles' weights.
//   quant_kernel     FP32 head scales from the maxima; K/V tiles (bulk-copied) ->
//                    blobs and 128-row Q blocks (GQA-packed) -> Q blobs, each
//                    assembled in shared memory and written with 16-byte stores.
//                    When pass 1 quantizes the K/V tiles inside its own launch
//                    (quant_role in quant_tile.cuh), only the Q blocks run here.
#include "apa_internal.h"
#include "quant_tile.cuh"
#include "tc.cuh"

namespace apa {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t ord_enc(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord_dec(uint32_t e) {
  return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}
// One elected thread brings rows [j0, j0 + nk) of the K and V slices of a tile
// into shared memory with two bulk copies (rows are 2d bytes, a multiple of 16;
// the slices start on 16-byte boundaries).  Every thread then waits, bounded;
// false if the wait gave up (the error word is set).
__device__ __forceinline__ bool load_kv_tile(uint16_t* ks, uint16_t* vs, const uint16_t* k, const uint16_t* v,
                                             int nk, int d, uint64_t* bar, int* err) {
  const uint32_t b = smem_u32(bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)nk * d * 2;
    mbar_arrive_expect_tx(b, 2 * bytes);
    bulk_g2s(smem_u32(ks), k, bytes, b);
    bulk_g2s(smem_u32(vs), v, bytes, b);
  }
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(b, 0)) {
    if (clock64() - t0 > APA_WAIT_LIMIT_CYCLES) {
      if (err) atomicCAS(err, 0, APA_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  __syncthreads();
  return v;  // valid in warp 0
}

__device__ __forceinline__ float absmax8(uint4 val) {
  const uint32_t w[4] = {val.x, val.y, val.z, val.w};
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16f(w[e] & 0xFFFF)), fabsf(bf16f(w[e] >> 16))));
  return m;
}

__global__ void __launch_bounds__(kThreads) stats_kernel(Shape s, const uint16_t* __restrict__ q,
                                                          const uint16_t* __restrict__ k,
                                                          const uint16_t* __restrict__ v, Workspace ws,
                                                          int n_kv_blocks, int q_rows_per_block, int do_kv,
                                                          int* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red[32];
  __shared__ __align__(8) uint64_t bar;
  const int d = s.d, T = s.T();
  if (do_kv && (int)blockIdx.x < n_kv_blocks) {
    const int bh = blockIdx.x / T, t = blockIdx.x % T;
    const int j0 = t * kTile, nk = min(kTile, s.Nkv - j0);
    const size_t base = kv_tile_offset(s, bh, t, err);
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem);
    uint16_t* vs = ks + kTile * d;
    if (!load_kv_tile(ks, vs, k + base, v + base, nk, d, &bar, err)) return;
    // max |V| over the tile
    float vm = 0.f;
    for (int i = threadIdx.x; i < nk * d / 8; i += blockDim.x) vm = fmaxf(vm, absmax8(reinterpret_cast<const uint4*>(vs)[i]));
    // per channel: FP32 sum over the tile's keys in ascending order, min, max
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      float acc = 0.f, mn = INFINITY, mx = -INFINITY;
#pragma unroll 8
      for (int j = 0; j < nk; ++j) {
        const float x = bf16f(ks[j * d + c]);
        acc = __fadd_rn(acc, x);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
      ws.ksum[((size_t)bh * T + t) * d + c] = acc;
      atomicMin(&ws.kmin[(size_t)bh * d + c], ord_enc(mn));
      atomicMax(&ws.kmax[(size_t)bh * d + c], ord_enc(mx));
    }
    // value norm of each key (value-weighted hot test): FP32 squares summed in channel
    // order, correctly rounded square root; the last two warps, one key per thread
    __shared__ float nrm[kTile];
    const int jn = threadIdx.x - (kThreads - kTile);
    if (ws.wv && jn >= 0 && jn < nk) {
      const uint4* row = reinterpret_cast<const uint4*>(vs + jn * d);
      float acc = 0.f;
      for (int c8 = 0; c8 < d / 8; ++c8) {
        const uint4 x = row[c8];
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = bf16f(w4[e] & 0xFFFF), hi = bf16f(w4[e] >> 16);
          acc = __fadd_rn(acc, __fmul_rn(lo, lo));
          acc = __fadd_rn(acc, __fmul_rn(hi, hi));
        }
      }
      nrm[jn] = __fsqrt_rn(acc);
    }
    vm = block_max(vm, red);  // (its barriers also publish nrm)
    if (threadIdx.x == 0) atomicMax(&ws.vamax[bh], __float_as_uint(vm));
    if (ws.wv && threadIdx.x == 32) {
      // the tile's largest norm and its FP32 norm sum in key order
      float a = 0.f, sum = 0.f;
      for (int j = 0; j < nk; ++j) {
        a = fmaxf(a, nrm[j]);
        sum = __fadd_rn(sum, nrm[j]);
      }
      ws.wv[(size_t)bh * T + t] = a;
      ws.vtsum[(size_t)bh * T + t] = sum;
    }
    return;
  }
  // max |Q| over a chunk of rows of one query head
  const int qb = blockIdx.x - (do_kv ? n_kv_blocks : 0);
  const int chunks_per_head = (s.Nq + q_rows_per_block - 1) / q_rows_per_block;
  const int bhq = qb / chunks_per_head, ch = qb % chunks_per_head;
  const int r0 = ch * q_rows_per_block, nr = min(q_rows_per_block, s.Nq - r0);
  const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)bhq * s.Nq + r0) * d);
  float qm = 0.f;
  for (int i = threadIdx.x; i < nr * d / 8; i += blockDim.x) qm = fmaxf(qm, absmax8(src[i]));
  qm = block_max(qm, red);
  if (threadIdx.x == 0) atomicMax(&ws.qamax[bhq], __float_as_uint(qm));
}

// Key mean per channel from the tile sums, in the pinned order: FP64 sums over
// ranges of kMeanRange consecutive tiles (ascending), then the range sums in
// ascending order.  One block per (b, KV head, 8 channels): 32 lanes per channel
// sum different ranges in parallel, one lane per channel adds the range sums.
// Also the maximum |k - mu| of the head (atomic max on the float bits).
constexpr int kMeanRange = 64;
constexpr int kRangesPerPass = 64;
constexpr int kFinChannels = 8;

// The head's mean key value norm in the key mean's order (FP64 sums of the FP32
// tile sums per range of kMeanRange tiles, then of the ranges), rounded to FP32,
// and each tile's weight = its largest norm / the mean (1 when the mean is 0).
__device__ void value_weights(const Shape& s, const Workspace& ws, int bh) {
  __shared__ double rs[kThreads];
  __shared__ float nbar_s;
  const int T = s.T(), nR = (T + kMeanRange - 1) / kMeanRange;
  const float* ts = ws.vtsum + (size_t)bh * T;
  double S = 0.0;
  for (int r0 = 0; r0 < nR; r0 += kThreads) {
    const int r = r0 + threadIdx.x;
    if (r < nR) {
      double Sr = 0.0;
      for (int t = r * kMeanRange; t < min(T, (r + 1) * kMeanRange); ++t) Sr += (double)ts[t];
      rs[threadIdx.x] = Sr;
    }
    __syncthreads();
    if (threadIdx.x == 0)
      for (int i = 0; i < min(kThreads, nR - r0); ++i) S += rs[i];
    __syncthreads();
  }
  if (threadIdx.x == 0) nbar_s = __double2float_rn(S / (double)s.Nkv);
  __syncthreads();
  const float nbar = nbar_s;
  float* w = ws.wv + (size_t)bh * T;
  for (int t = threadIdx.x; t < T; t += kThreads) w[t] = nbar == 0.f ? 1.f : __fdiv_rn(w[t], nbar);
}

__global__ void __launch_bounds__(kThreads) finalize_kernel(Shape s, Workspace ws) {
  __shared__ double rs[kRangesPerPass][kFinChannels];
  const int cblocks = s.d / kFinChannels;
  if ((int)blockIdx.x >= s.BH() * cblocks) {  // one extra block per head when value-weighted
    value_weights(s, ws, blockIdx.x - s.BH() * cblocks);
    return;
  }
  const int bh = blockIdx.x / cblocks, cl = threadIdx.x % kFinChannels, lane = threadIdx.x / kFinChannels;
  constexpr int kLanes = kThreads / kFinChannels;
  const int c = (blockIdx.x % cblocks) * kFinChannels + cl;
  const int d = s.d, T = s.T(), nR = (T + kMeanRange - 1) / kMeanRange;
  const float* col = ws.ksum + (size_t)bh * T * d + c;
  double S = 0.0;
  for (int r0 = 0; r0 < nR; r0 += kRangesPerPass) {
    for (int r = r0 + lane; r < min(nR, r0 + kRangesPerPass); r += kLanes) {
      const int t0 = r * kMeanRange, t1 = min(T, t0 + kMeanRange);
      double Sr = 0.0;
      for (int t = t0; t < t1; t += 16) {
        float x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = t + u < t1 ? col[(size_t)(t + u) * d] : 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (t + u < t1) Sr += (double)x[u];
      }
      rs[r - r0][cl] = Sr;
    }
    __syncthreads();
    if (lane == 0)
      for (int r = 0; r < min(kRangesPerPass, nR - r0); ++r) S += rs[r][cl];
    __syncthreads();
  }
  if (lane == 0) {
    const float mu = __double2float_rn(S / (double)s.Nkv);
    ws.mu[(size_t)bh * d + c] = mu;
    const float mn = ord_dec(ws.kmin[(size_t)bh * d + c]), mx = ord_dec(ws.kmax[(size_t)bh * d + c]);
    float am = fmaxf(fabsf(__fsub_rn(mx, mu)), fabsf(__fsub_rn(mn, mu)));
    // the kFinChannels lane-0 threads are lanes 0..7 of warp 0
#pragma unroll
    for (int o = kFinChannels / 2; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0x000000FFu, am, o));
    if (cl == 0) atomicMax(&ws.kcamax[bh], __float_as_uint(am));
  }
}

__global__ void __launch_bounds__(kThreads) quant_kernel(Shape s, const uint16_t* __restrict__ q,
                                                          const uint16_t* __restrict__ k,
                                                          const uint16_t* __restrict__ v, Workspace ws,
                                                          int n_kv_blocks, int do_kv, int* err, int lse,
                                                          int kv_scales_from_q) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  const int d = s.d, T = s.T();
  if (do_kv && (int)blockIdx.x < n_kv_blocks) {
    const int bh = blockIdx.x / T, t = blockIdx.x % T;
    const int j0 = t * kTile, nk = min(kTile, s.Nkv - j0);
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem);
    uint16_t* vs = ks + kTile * d;
    uint8_t* img = reinterpret_cast<uint8_t*>(vs + kTile * d);  // the blob, assembled here
    float* mus = reinterpret_cast<float*>(img + blob_bytes(d));
    const size_t base = kv_tile_offset(s, bh, t, err);
    // keys past Nkv quantize as zero V; the image starts zeroed (padding included)
    for (int i = threadIdx.x; i < (kTile - nk) * d / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(vs + nk * d)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < blob_bytes(d) / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(img)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int c = threadIdx.x; c < d; c += blockDim.x) mus[c] = ws.mu[(size_t)bh * d + c];
    if (!load_kv_tile(ks, vs, k + base, v + base, nk, d, &bar, err)) return;
    __syncthreads();
    // FP32 head scales from the head maxima (the head's largest magnitude maps to 2688)
    const float sk = head_scale(__uint_as_float(ws.kcamax[bh])), sv = head_scale(__uint_as_float(ws.vamax[bh]));
    if (t == 0 && threadIdx.x == 0) {
      ws.s_k[bh] = sk;
      ws.s_v[bh] = sv;
    }
    quant_kv_tile(s, ws, bh, t, nk, ks, vs, mus, img, lse != 0, threadIdx.x, blockDim.x);
    __syncthreads();
    store_image(ws.kv_blob + ((size_t)bh * T + t) * blob_bytes(d), img, blob_bytes(d));
    return;
  }
  // Q: one 128-row block of packed rows p = pos*G + g
  const int qb = blockIdx.x - (do_kv ? n_kv_blocks : 0);
  const int nblk = s.nblk(), G = s.G(), R = s.R();
  const int bh = qb / nblk, blk = qb % nblk;
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  uint8_t* img = smem;
  uint8_t* img2 = smem + qblob_bytes(d);  // the residual term, when asked for
  const bool q2 = ws.q2_blob != nullptr;
  if (blk == 0 && kv_scales_from_q && threadIdx.x == 0) {
    // the K/V tiles are quantized inside the pass-1 launch, which needs the head
    // scales from its start: the Q blocks publish them
    ws.s_k[bh] = head_scale(__uint_as_float(ws.kcamax[bh]));
    ws.s_v[bh] = head_scale(__uint_as_float(ws.vamax[bh]));
  }
  if (blk == 0)
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      const int hq = b * s.Hq + h * G + g;
      ws.s_q[hq] = head_scale(__uint_as_float(ws.qamax[hq]));
    }
  const int ncb = d / 16;
  for (int it = threadIdx.x; it < kBlockRows * ncb; it += blockDim.x) {
    const int p = it / ncb, cb = it % ncb, P = blk * kBlockRows + p;
    uint2 codes = make_uint2(0u, 0u), codes2 = make_uint2(0u, 0u);
    uint32_t sb = 0, sb2 = 0;
    if (P < R) {
      const int g = P % G, pos = P / G, hq = b * s.Hq + h * G + g;
      const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)hq * s.Nq + pos) * d + cb * 16);
      const uint4 a0 = src[0], a1 = src[1];
      const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16f(w[i] & 0xFFFF);
        x[2 * i + 1] = bf16f(w[i] >> 16);
      }
      const float sq = head_scale(__uint_as_float(ws.qamax[hq]));
      sb = quant16_mode(x, sq, &codes, lse);
      if (q2) {
        // the FP4 residual in the same head scale: r = fp32(x - fp32(E2M1 * UE4M3 * s))
        // (the product of a code and a scale has at most 7 significant bits: exact)
        const float sv1 = ue4m3_value(sb);
        float r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t c = ((i < 8 ? codes.x >> (4 * i) : codes.y >> (4 * (i - 8)))) & 0xFu;
          r[i] = __fsub_rn(x[i], __fmul_rn(e2m1_value(c) * sv1, sq));
        }
        sb2 = quant16_mode(r, sq, &codes2, lse);
      }
    }
    *reinterpret_cast<uint2*>(img + fp4_kmajor_off(p, cb, d / 2)) = codes;
    img[qblob_sf(d) + (cb >> 2) * 512 + sf_atom_off(p, cb & 3)] = (uint8_t)sb;
    if (q2) {
      *reinterpret_cast<uint2*>(img2 + fp4_kmajor_off(p, cb, d / 2)) = codes2;
      img2[qblob_sf(d) + (cb >> 2) * 512 + sf_atom_off(p, cb & 3)] = (uint8_t)sb2;
    }
  }
  __syncthreads();
  store_image(ws.q_blob + ((size_t)bh * nblk + blk) * qblob_bytes(d), img, qblob_bytes(d));
  if (q2) store_image(ws.q2_blob + ((size_t)bh * nblk + blk) * qblob_bytes(d), img2, qblob_bytes(d));
}

// The all-exact path (eps = 0) runs P.V as one FP16 term against an FP16 copy
// of V, the same copy the quantizer writes in APA mode: V divided by the head's
// power-of-two scale v16_scale(max |v|), which is 1 unless max |v| > 2^15.  One
// pass converts every head with divisor 1 and takes the head maxima; a second,
// per block, re-converts its keys only if its head needs a divisor (it then also
// overwrites what the first pass may have saturated).  Blocks take kV16Tiles key
// tiles of one head.
constexpr int kV16Tiles = 4;

__device__ __forceinline__ uint4 v16_of(uint4 val, float inv) {
  const uint32_t w[4] = {val.x, val.y, val.z, val.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = cvt_f16x2(bf16f(w[e] & 0xFFFF) * inv, bf16f(w[e] >> 16) * inv);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// fixup = 0: the first pass; 1: the re-conversion of heads whose maximum needs a divisor.
__global__ void __launch_bounds__(kThreads) v16_kernel(Shape s, const uint16_t* __restrict__ v, Workspace ws,
                                                        int fixup, int* err) {
  __shared__ float red[32];
  const int bh = blockIdx.y, T = s.T(), d = s.d;
  float inv = 1.f;
  if (fixup) {
    const float sc = v16_scale(__uint_as_float(ws.vamax[bh]));
    if (sc == 1.f) return;
    inv = 1.f / sc;
  }
  float vm = 0.f;
  for (int t = blockIdx.x * kV16Tiles; t < min(T, (int)(blockIdx.x + 1) * kV16Tiles); ++t) {
    const int nk = min(kTile, s.Nkv - t * kTile);
    const uint4* src = reinterpret_cast<const uint4*>(v + kv_tile_offset(s, bh, t, err));
    uint4* dst = reinterpret_cast<uint4*>(ws.v16 + ((size_t)bh * s.Nkv + (size_t)t * kTile) * d);
    for (int i = threadIdx.x; i < nk * d / 8; i += blockDim.x) {
      const uint4 val = src[i];
      if (!fixup) vm = fmaxf(vm, absmax8(val));
      dst[i] = v16_of(val, inv);
    }
  }
  if (!fixup) {
    vm = block_max(vm, red);
    if (threadIdx.x == 0) atomicMax(&ws.vamax[bh], __float_as_uint(vm));
  }
}

}  // namespace

cudaError_t launch_v16(const Shape& s, const void* v, const Workspace& ws, cudaStream_t st) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(ws.vamax, 0x00, sizeof(uint32_t) * s.BH(), st))) return e;
  const dim3 grid((s.T() + kV16Tiles - 1) / kV16Tiles, s.BH());
  int* err = device_error_word();
  for (int fixup = 0; fixup < 2; ++fixup) {
    v16_kernel<<<grid, kThreads, 0, st>>>(s, (const uint16_t*)v, ws, fixup, err);
    if ((e = cudaGetLastError())) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_quantize(const Shape& s, const void* q, const void* k, const void* v, const Workspace& ws,
                            bool do_q, bool do_kv, cudaStream_t st, bool lse, bool kv_in_pass1) {
  const int BH = s.BH(), d = s.d, T = s.T();
  int* err = device_error_word();
  cudaError_t e;
  if (do_kv) {
    if ((e = cudaMemsetAsync(ws.kmin, 0xFF, sizeof(uint32_t) * BH * d, st))) return e;
    if ((e = cudaMemsetAsync(ws.kmax, 0x00, sizeof(uint32_t) * BH * d, st))) return e;
    if ((e = cudaMemsetAsync(ws.vamax, 0x00, sizeof(uint32_t) * BH, st))) return e;
    if ((e = cudaMemsetAsync(ws.kcamax, 0x00, sizeof(uint32_t) * BH, st))) return e;
  }
  if (do_q && (e = cudaMemsetAsync(ws.qamax, 0x00, sizeof(uint32_t) * s.B * s.Hq, st))) return e;
  if (kv_in_pass1 && (e = cudaMemsetAsync(ws.kv_ready, 0x00, sizeof(uint32_t) * ((size_t)BH * T + 1), st)))
    return e;
  const int n_kv = do_kv ? BH * T : 0;
  const int q_rows = 64;
  const int n_q = do_q ? s.B * s.Hq * ((s.Nq + q_rows - 1) / q_rows) : 0;
  const size_t sm1 = (size_t)kTile * d * 2 * 2;
  if (sm1 > 48 * 1024 &&
      (e = cudaFuncSetAttribute(stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)))
    return e;
  if (n_kv + n_q > 0)
    stats_kernel<<<n_kv + n_q, kThreads, sm1, st>>>(s, (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, ws,
                                                    n_kv, q_rows, do_kv, err);
  if ((e = cudaGetLastError())) return e;
  if (do_kv) {
    finalize_kernel<<<BH * (d / kFinChannels) + (ws.wv ? BH : 0), kThreads, 0, st>>>(s, ws);
    if ((e = cudaGetLastError())) return e;
  }
  const int n_qb = do_q ? BH * s.nblk() : 0;
  const int n_kvq = kv_in_pass1 ? 0 : n_kv;  // K/V blocks of the quantizer kernel
  const size_t sm2 = (size_t)kTile * d * 2 * 2 + blob_bytes(d) + d * 4;
  if (sm2 > 48 * 1024 &&
      (e = cudaFuncSetAttribute(quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)))
    return e;
  if (n_kvq + n_qb > 0)
    quant_kernel<<<n_kvq + n_qb, kThreads, sm2, st>>>(s, (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v,
                                                      ws, n_kvq, n_kvq > 0, err, lse ? 1 : 0, kv_in_pass1 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace apa
