// quant_tile.cuh -- the NVFP4 block quantizer of one 16-value block and of one
// 64-key K/V tile, shared by the standalone quantizer kernel and the K/V
// quantizer role that runs inside the pass-1 launch.
//
// "APA: sloppy attention, exact where it counts" (rfriedmann.de blog),
// "Pass 1: FP4 everywhere, with a hot test" and "A 9216-byte blob per tile".
// Bit-exact by construction: every FP32 operation is an explicitly rounded
// intrinsic (no contraction); the op order per block is stated at quant16.
#pragma once
#include "apa_internal.h"
#include "tc.cuh"

namespace apa {
namespace {

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  uint32_t E = code >> 3, m = code & 7;
  if (E == 0) return (float)m * 0.001953125f;  // m * 2^-9
  return __uint_as_float(((E + 120u) << 23) | (m << 20));
}
// Value of a 4-bit E2M1 code (sign in bit 3): 0, 0.5, 1, 1.5, 2, 3, 4, 6.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  const float v = m < 4 ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1)) * (1.f + 0.5f * (float)(m & 1u));
  return (c & 8u) ? -v : v;
}
__device__ __forceinline__ float head_scale(float amax) { return amax == 0.f ? 1.f : __fdiv_rn(amax, 2688.f); }

// Quantizes 16 values with head scale s; returns the scale code, writes 8 code bytes.
__device__ __forceinline__ uint32_t quant16(const float* x, float s, uint2* codes) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
  const float r = __fdiv_rn(a, __fmul_rn(6.f, s));
  const uint32_t sb = cvt_ue4m3(r);
  if (sb == 0) {
    *codes = make_uint2(0u, 0u);
    return 0;
  }
  const float inv = __frcp_rn(__fmul_rn(ue4m3_value(sb), s));
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = cvt_e2m1x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
    w[i >> 2] |= byte << (8 * (i & 3));
  }
  *codes = make_uint2(w[0], w[1]);
  return sb;
}

// E2M1 codes of 16 values under scale code sb, and the FP32 sum of squared
// errors sum_i fp32(x_i - fp32(E2M1(code_i) * D))^2 in index order.
__device__ __forceinline__ float block_codes(const float* x, float s, uint32_t sb, uint2* codes) {
  const float D = __fmul_rn(ue4m3_value(sb), s);
  const float inv = __frcp_rn(D);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t byte = cvt_e2m1x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
    w[i >> 2] |= byte << (8 * (i & 3));
  }
  float err = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t c = (w[i >> 3] >> (4 * (i & 7))) & 0xFu;
    const float t = __fsub_rn(x[i], __fmul_rn(e2m1_value(c), D));
    err = __fadd_rn(err, __fmul_rn(t, t));
  }
  *codes = make_uint2(w[0], w[1]);
  return err;
}

// quant16 with, when lse is set, the block scale picked by least squared error
// among the nearest code and its two neighbours (tried in that order; only a
// strictly smaller error replaces the pick).
__device__ __forceinline__ uint32_t quant16_mode(const float* x, float s, uint2* codes, bool lse) {
  uint32_t sb = quant16(x, s, codes);
  if (!lse || sb == 0) return sb;
  const uint32_t nearest = sb;
  float best = block_codes(x, s, nearest, codes);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t c = j == 0 ? nearest - 1 : nearest + 1;
    if (c < 1 || c > 0x7E) continue;
    uint2 c2;
    const float e = block_codes(x, s, c, &c2);
    if (e < best) {
      best = e;
      sb = c;
      *codes = c2;
    }
  }
  return sb;
}

// Copies a blob image from shared memory to global memory with 16-byte stores
// (threads tid = 0 .. nth-1).
__device__ __forceinline__ void store_image(uint8_t* dst, const uint8_t* img, int bytes, int tid, int nth) {
  for (int i = tid; i < bytes / 16; i += nth)
    reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(img)[i];
}
__device__ __forceinline__ void store_image(uint8_t* dst, const uint8_t* img, int bytes) {
  store_image(dst, img, bytes, threadIdx.x, blockDim.x);
}

// Barrier over the nth threads of a group (named barrier id, 1..4); the _and
// form also returns whether v held in every thread of the group.  The ids are
// immediates, so a kernel reserves only the barriers it can name.
template <int kId>
__device__ __forceinline__ void bar_sync_id(int nth) {
  asm volatile("bar.sync %0, %1;" ::"n"(kId), "r"(nth) : "memory");
}
template <int kId>
__device__ __forceinline__ bool bar_red_and_id(int nth, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.and.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kId), "r"(nth)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void group_sync(int id, int nth) {
  switch (id) {
    case 1: bar_sync_id<1>(nth); break;
    case 2: bar_sync_id<2>(nth); break;
    case 3: bar_sync_id<3>(nth); break;
    default: bar_sync_id<4>(nth); break;
  }
}
__device__ __forceinline__ bool group_sync_and(int id, int nth, bool v) {
  switch (id) {
    case 1: return bar_red_and_id<1>(nth, v);
    case 2: return bar_red_and_id<2>(nth, v);
    case 3: return bar_red_and_id<3>(nth, v);
    default: return bar_red_and_id<4>(nth, v);
  }
}

// Quantizes the tile of keys [t*64, t*64 + nk) of head bh whose K and V rows are
// in shared memory (ks, vs: 64 rows x d bf16; V rows past nk zero) into the blob
// image img (zeroed by the caller), centring K by the key mean mus (d floats in
// shared memory), and writes the tile's FP16 V rows when ws.v16 is set.  Threads
// tid = 0 .. nth-1 of a group take part; nth is a multiple of d / 16.
__device__ __forceinline__ void quant_kv_tile(const Shape& s, const Workspace& ws, int bh, int t, int nk,
                                              const uint16_t* ks, const uint16_t* vs, const float* mus,
                                              uint8_t* img, bool lse, int tid, int nth) {
  const int d = s.d;
  const size_t base = ((size_t)bh * s.Nkv + (size_t)t * kTile) * d;
  // FP32 head scales from the head maxima (the head's largest magnitude maps to 2688)
  const float sk = head_scale(__uint_as_float(ws.kcamax[bh])), sv = head_scale(__uint_as_float(ws.vamax[bh]));
  const int ncb = d / 16;
  // K: per (key n, 16-channel block cb), centred.  nth is a multiple of ncb,
  // so each thread keeps one cb and its 16 means in registers.
  {
    const int cb = tid % ncb;
    float mu16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) mu16[i] = mus[cb * 16 + i];
    for (int n = tid / ncb; n < nk; n += nth / ncb) {
      const uint4* src = reinterpret_cast<const uint4*>(ks + n * d + cb * 16);
      const uint4 a0 = src[0], a1 = src[1];
      const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = __fsub_rn(bf16f(w[i] & 0xFFFF), mu16[2 * i]);
        x[2 * i + 1] = __fsub_rn(bf16f(w[i] >> 16), mu16[2 * i + 1]);
      }
      uint2 codes;
      const uint32_t sb = quant16_mode(x, sk, &codes, lse);
      *reinterpret_cast<uint2*>(img + blob_kcodes(d) + fp4_kmajor_off(n, cb, d / 2)) = codes;
      const int kb = cb >> 2, k16 = cb & 3;
      img[blob_ksf(d) + (kb >> 1) * 512 + (n & 31) * 16 + ((n >> 5) + 2 * (kb & 1)) * 4 + k16] = (uint8_t)sb;
    }
  }
  // V^T: per (channel pair, 16-key block kb16)
  for (int it = tid; it < (d / 2) * 4; it += nth) {
    const int cp = it % (d / 2), kb16 = it / (d / 2);
    float x0[16], x1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = reinterpret_cast<const uint32_t*>(vs + (kb16 * 16 + i) * d)[cp];
      x0[i] = bf16f(w & 0xFFFF);
      x1[i] = bf16f(w >> 16);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = 2 * cp + e;
      uint2 codes;
      const uint32_t sb = quant16_mode(e ? x1 : x0, sv, &codes, lse);
      *reinterpret_cast<uint2*>(img + blob_vcodes(d) + fp4_kmajor_off(c, kb16, 32)) = codes;
      img[blob_vsf(d) + (c >> 7) * 512 + sf_atom_off(c & 127, kb16)] = (uint8_t)sb;
    }
  }
  // FP16 copy of the tile's V rows for pass 2, divided by the head's power-of-two scale
  if (ws.v16) {
    const float inv = 1.f / v16_scale(__uint_as_float(ws.vamax[bh]));
    uint4* dst = reinterpret_cast<uint4*>(ws.v16 + base);
    for (int i = tid; i < nk * d / 8; i += nth) {
      const uint4 val = reinterpret_cast<const uint4*>(vs)[i];
      const uint32_t w[4] = {val.x, val.y, val.z, val.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = cvt_f16x2(bf16f(w[e] & 0xFFFF) * inv, bf16f(w[e] >> 16) * inv);
      dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Bytes of shared memory one group of the K/V quantizer role needs: nbuf K/V tile
// buffers, the blob image, the key mean and two mbarriers (a multiple of 16).
__host__ __device__ constexpr int quant_role_smem(int d, int nbuf = 2) {
  return nbuf * 2 * kTile * d * 2 + blob_bytes(d) + d * 4 + 16;
}

constexpr int kQuantRoleGroups = 4;  // at most, per block

// The K/V quantizer as one role of a larger cooperative kernel, run by a group
// of nth threads (tid = 0 .. nth-1, named barrier group + 1; the groups of a
// block work independently).  The group takes tickets from *ticket, one
// (step, head) each: step 0 is tile 0, step i is tile T - i, every head at each
// step, which is the order in which pass 1 visits the tiles ("Tile order": the
// sink, then back from the causal diagonal).  It quantizes the tile, stores its
// blob and FP16 V rows, and then publishes ready[bh * T + t] = 1 (release at GPU
// scope) for pass 1 to wait on.  With nbuf = 2 the K/V loads are double-buffered:
// the next ticket's bulk copies fly while the group quantizes the current tile;
// with nbuf = 1 they are issued once the tile is done.  `smem` (16-byte aligned)
// holds quant_role_smem(d, nbuf) bytes of the group's own.  Returns false if a
// wait gave up (the error word is set).
__device__ __noinline__ bool quant_role(const Shape& s, const uint16_t* __restrict__ k,
                                        const uint16_t* __restrict__ v, const Workspace& ws, uint32_t* ready,
                                        uint32_t* ticket, bool lse, uint8_t* smem, int* err, int group, int tid,
                                        int nth, int nbuf) {
  __shared__ int tk_all[kQuantRoleGroups][2];
  int* tk_s = tk_all[group];
  const int bid = 1 + group;
  const int d = s.d, T = s.T(), BH = s.BH(), total = BH * T;
  const int kvb = kTile * d * 2;  // bytes of one K or V tile
  uint8_t* img = smem + 2 * nbuf * kvb;
  float* mus = reinterpret_cast<float*>(img + blob_bytes(d));
  const uint32_t bar0 = smem_u32(mus + d);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init();
    tk_s[0] = (int)atomicAdd(ticket, 1u);
  }
  group_sync(bid, nth);
  auto tile_of = [&](int tk, int* bh) {
    *bh = tk % BH;
    const int step = tk / BH;
    return step == 0 ? 0 : T - step;
  };
  // tid 0: the bulk copies of ticket tk's K and V rows into buffer buf
  auto issue = [&](int tk, int buf) {
    int bh;
    const int t = tile_of(tk, &bh);
    const int nk = min(kTile, s.Nkv - t * kTile);
    const size_t base = kv_tile_offset(s, bh, t, err);
    const uint32_t bytes = (uint32_t)nk * d * 2, bar = bar0 + 8u * buf;
    const uint32_t dst = smem_u32(smem + 2 * kvb * buf);
    fence_proxy_async_smem();  // the group's earlier accesses of this buffer come first
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(dst, k + base, bytes, bar);
    bulk_g2s(dst + kvb, v + base, bytes, bar);
  };
  int cur = tk_s[0];
  if (tid == 0 && cur < total) issue(cur, 0);
  uint32_t parity = 0;                       // bit b: the phase buffer b waits for next
  uint32_t pending = cur < total ? 1u : 0u;  // bit b: buffer b has copies in flight (tid 0's view)
  int buf = 0;
  bool ok = true;
  for (int j = 0; cur < total; ++j) {
    int bh;
    const int t = tile_of(cur, &bh);
    const int nk = min(kTile, s.Nkv - t * kTile);
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem + 2 * kvb * buf);
    uint16_t* vs = ks + kTile * d;
    if (tid == 0) {
      const int nx = (int)atomicAdd(ticket, 1u);
      tk_s[(j + 1) & 1] = nx;
      if (nx < total && nbuf == 2) {
        issue(nx, buf ^ 1);
        pending |= 1u << (buf ^ 1);
      }
    }
    // V rows past the last key quantize as zero; the image starts zeroed
    for (int i = tid; i < (kTile - nk) * d / 8; i += nth)
      reinterpret_cast<uint4*>(vs + nk * d)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < blob_bytes(d) / 16; i += nth) reinterpret_cast<uint4*>(img)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int c = tid; c < d; c += nth) mus[c] = ws.mu[(size_t)bh * d + c];
    {
      const uint32_t bar = bar0 + 8u * buf, par = (parity >> buf) & 1u;
      const unsigned long long t0 = clock64();
      while (ok && !mbar_try_wait(bar, par))
        if (clock64() - t0 > APA_WAIT_LIMIT_CYCLES) {
          if (err) atomicCAS(err, 0, APA_DEVERR_TIMEOUT);
          ok = false;
        }
      if (ok) {
        parity ^= 1u << buf;
        pending &= ~(1u << buf);
      }
    }
    ok = group_sync_and(bid, nth, ok);
    const int nxt = tk_s[(j + 1) & 1];
    if (!ok) break;
    quant_kv_tile(s, ws, bh, t, nk, ks, vs, mus, img, lse, tid, nth);
    group_sync(bid, nth);
    store_image(ws.kv_blob + ((size_t)bh * T + t) * blob_bytes(d), img, blob_bytes(d), tid, nth);
    group_sync(bid, nth);
    if (tid == 0) {
      __threadfence();
      st_release_gpu(ready + (size_t)bh * T + t, 1u);
      if (nbuf == 1 && nxt < total) {  // the only buffer is free again
        issue(nxt, 0);
        pending |= 1u;
      }
    }
    cur = nxt;
    if (nbuf == 2) buf ^= 1;
  }
  if (!ok && tid == 0) {
    // let the copies in flight land before the block's shared memory goes away (bounded)
    for (int b = 0; b < 2; ++b) {
      if (!((pending >> b) & 1u)) continue;
      const uint32_t bar = bar0 + 8u * b, par = (parity >> b) & 1u;
      const unsigned long long t0 = clock64();
      while (!mbar_try_wait(bar, par) && clock64() - t0 <= APA_WAIT_LIMIT_CYCLES) {
      }
    }
  }
  return ok;
}

}  // namespace
}  // namespace apa
