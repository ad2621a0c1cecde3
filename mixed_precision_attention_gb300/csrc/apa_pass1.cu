// apa_pass1.cu -- pass 1: every key tile in block-scaled NVFP4, with the hot test.
//
// "APA: sloppy attention, exact where it counts" (rfriedmann.de blog),
// "Pass 1: FP4 everywhere, with a hot test", per tile and 16-row group:
//   1. S = Q K^T on the FP4 tensor cores, causal mask applied;
//   2. P directly in FP4: each 16-key group gets its own scale, folded into
//      the exponent bias, so ex2 produces the quantized P;
//   3. row sums l_t from the same P, via one extra MMA against an E2M1 ones tile;
//   4. the hot test: if any of the group's 16 rows has l_t > eps * lambda, the
//      tile is hot: set the mask bit, skip the PV product for the group;
//   5. cold tiles accumulate o += P V in FP4, the cold row sum grows by l_t.
// Tile order: tile 0 (the sink), then from the causal diagonal backwards
// ("Tile order").  Frames: lazy maximum with tau = 4 ("Lazy maximum"); a hot
// tile lifts the frame only to max(m, c - 32) ("The bug: a sink that drowned
// the tail", the decoupled cold frame); the P group scale is UE4M3 ("Second
// hunt") clamped at 2^-6 ("The bug").  lambda is the running FP4 sum over every
// tile judged so far, hot ones included ("Cold verdicts are safe").
//
// GB300 design: one CTA = one 128-row block of GQA-packed rows of one KV head.
//   warps 0-3  one thread per row (TMEM lane = row): group maxima, frame, P
//              encode (ex2 + cvt.e2m1x2), P to shared memory, P scales to TMEM
//              (tcgen05.st), hot vote (ballot over the 16 lanes of a group),
//              frame / lambda / l commit, O rescale when the frame moves;
//   warp 4     bulk-copy producer: the Q blob, then one 72*d-byte NVFP4 blob per
//              tile (K codes, V^T codes and both scale sets) into a 4-stage ring;
//   warp 5     TMEM owner and MMA issuer (tcgen05.mma kind::mxf4nvf4,
//              scale_vec::4X): S (M128 N64), ones (M128 N16), PV (M128 N=d), the
//              scale copies (tcgen05.cp), and the block's hot-tile list.
// At d <= 128 a CTA uses 256 TMEM columns and ~55 KB of shared memory, so two
// CTAs share an SM and hide each other's softmax-to-MMA round trips.
#include "apa_internal.h"
#include "tc.cuh"

namespace apa {

namespace {

struct P1Params {
  Shape s;
  const uint8_t* kv_blob;
  const uint8_t* q_blob;
  const float* s_k;
  const float* s_v;
  const float* s_q;
  float eps;
  float* state_o;
  float2* state_ml;
  uint32_t* hot_list;
  uint32_t* hot_count;
  uint32_t* hot_mask;  // may be null
  int* err;
};

constexpr int kThreads = 192;

template <int D>
struct P1Cfg {
  static constexpr int NS = 4;
  static constexpr int kBlob = blob_bytes(D);
  static constexpr int kQBlob = qblob_bytes(D);
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = (kQBlob + 1023) / 1024 * 1024;
  static constexpr int kPOff = kStageOff + NS * kBlob;  // 2 x (128 rows x 32 B)
  static constexpr int kOnesOff = kPOff + 2 * 4096;     // 16 rows x 32 B of E2M1 1.0
  static constexpr int kOnesSfOff = kOnesOff + 512;     // 512-B scale atom of UE4M3 1.0
  static constexpr int kSmem = kOnesSfOff + 512 + 128;
  static constexpr uint32_t kTmemCols = D <= 128 ? 256 : 512;
  static constexpr uint32_t kO = 0, kS = D, kL = D + 64, kSFQ = D + 80;
  static constexpr uint32_t kSFK = kSFQ + 4 * (D / 64);      // 2 buffers of 4 * sf_chunks(D)
  static constexpr uint32_t kSFV = kSFK + 8 * sf_chunks(D);  // 2 buffers of 4 * sf_chunks(D)
  static constexpr uint32_t kSFP = kSFV + 8 * sf_chunks(D);  // 2 buffers of 4
  static constexpr uint32_t kSFO = kSFP + 8;
  static_assert(kSFO + 4 <= kTmemCols, "TMEM budget");
};

__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, int* err) {
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > APA_WAIT_LIMIT_CYCLES) {
      if (err) atomicCAS(err, 0, APA_DEVERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ float ue4m3_value(uint32_t code) {
  const uint32_t E = code >> 3, m = code & 7;
  if (E == 0) return (float)m * 0.001953125f;
  return __uint_as_float(((E + 120u) << 23) | (m << 20));
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, (D <= 128 ? 2 : 1)) pass1_kernel(const P1Params p) {
  using C = P1Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  // barriers: q_full, blob_full[4], blob_empty[4], s_full, s_free, p_full[2], l_full, dec[2], pv_done[2], drain
  __shared__ __align__(8) uint64_t bars[18];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t gbits[2][4];

  const Shape& s = p.s;
  const int nblk = s.nblk(), BH = s.BH(), G = s.G(), R = s.R(), T = s.T(), off = s.off();
  const int bh = blockIdx.x % BH, blk = nblk - 1 - (int)(blockIdx.x / BH);
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  const int p0 = blk * kBlockRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  auto blob_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto blob_empty = [&](int st) { return bar0 + 8u * (5 + st); };
  const uint32_t s_full = bar0 + 8u * 9, s_free = bar0 + 8u * 10;
  auto p_full = [&](int b2) { return bar0 + 8u * (11 + b2); };
  const uint32_t l_full = bar0 + 8u * 13;
  auto dec = [&](int b2) { return bar0 + 8u * (14 + b2); };
  auto pv_done = [&](int b2) { return bar0 + 8u * (16 + b2); };
  // drain shares the last slot with nothing else
  __shared__ __align__(8) uint64_t drain_bar;
  const uint32_t drain = smem_u32(&drain_bar);
  auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool okl = mbar_wait(bar, parity, &abort_flag, p.err);
    return __all_sync(0xffffffffu, okl);
  };

  const int last_row = min(R, p0 + kBlockRows) - 1;
  const int t_hi = s.causal ? min(T - 1, (last_row / G + off) / kTile) : T - 1;
  const int n = t_hi + 1;
  auto tile_of = [&](int i) { return i == 0 ? 0 : t_hi + 1 - i; };
  const int n_valid_groups = (min(R, p0 + kBlockRows) - p0 + kGroupRows - 1) / kGroupRows;
  const uint32_t invalid_groups = 0xFFu & ~((1u << n_valid_groups) - 1u);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < 18; ++i) {
      const bool per_warp = (i == 10) || (i >= 11 && i <= 12) || (i >= 14 && i <= 15);  // s_free, p_full, dec
      mbar_init(bar0 + 8u * i, per_warp ? 4u : 1u);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // the ones tile (E2M1 1.0 = code 2) and its scale atom (UE4M3 1.0 = 0x38)
    reinterpret_cast<uint2*>(smem + C::kOnesOff)[threadIdx.x] =
        threadIdx.x < 64 ? make_uint2(0x22222222u, 0x22222222u) : make_uint2(0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ bulk-copy producer
    if (lane == 0) {
      const uint8_t* qsrc = p.q_blob + ((size_t)bh * nblk + blk) * C::kQBlob;
      mbar_arrive_expect_tx(q_full, C::kQBlob);
      bulk_g2s(sbase + C::kQOff, qsrc, C::kQBlob, q_full);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(blob_empty(st), ((i / C::NS) - 1) & 1, &abort_flag, p.err)) break;
        const uint8_t* src = p.kv_blob + ((size_t)bh * T + tile_of(i)) * C::kBlob;
        mbar_arrive_expect_tx(blob_full(st), C::kBlob);
        bulk_g2s(sbase + C::kStageOff + st * C::kBlob, src, C::kBlob, blob_full(st));
        issued = i + 1;
      }
      if (abort_flag) {
        wait_bounded(q_full, 0, p.err);
        for (int i = max(0, issued - C::NS); i < issued; ++i) wait_bounded(blob_full(i % C::NS), (i / C::NS) & 1, p.err);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_nvf4(128, 64), idL = idesc_nvf4(128, 16), idO = idesc_nvf4(128, D);
      uint32_t* list = p.hot_list + ((size_t)bh * nblk + blk) * T;
      uint32_t count = 0;
      bool ok = mbar_wait(q_full, 0, &abort_flag, p.err);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tmem_cp_32x128b_x4(tmem + C::kSFQ + 4 * a, smem_desc(sbase + C::kQOff + qblob_sf(D) + 512 * a, 128, 128, 0));
        tmem_cp_32x128b_x4(tmem + C::kSFO, smem_desc(sbase + C::kOnesSfOff, 128, 128, 0));
      }
      auto issue_s = [&](int i) -> bool {
        const int st = i % C::NS;
        if (!mbar_wait(blob_full(st), (i / C::NS) & 1, &abort_flag, p.err)) return false;
        if (i >= 1 && !mbar_wait(s_free, (i - 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t blob = sbase + C::kStageOff + st * C::kBlob;
        const uint32_t sfk = tmem + C::kSFK + 4 * sf_chunks(D) * (i & 1);
        const uint32_t sfv = tmem + C::kSFV + 4 * sf_chunks(D) * (i & 1);
#pragma unroll
        for (int c = 0; c < sf_chunks(D); ++c) {
          tmem_cp_32x128b_x4(sfk + 4 * c, smem_desc(blob + blob_ksf(D) + 512 * c, 128, 128, 0));
          tmem_cp_32x128b_x4(sfv + 4 * c, smem_desc(blob + blob_vsf(D) + 512 * c, 128, 128, 0));
        }
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk) {
          const uint64_t ad = smem_desc(sbase + C::kQOff + 256 * kk, 128, 4 * D, 0);
          const uint64_t bd = smem_desc(blob + blob_kcodes(D) + 256 * kk, 128, 4 * D, 0);
          mma_nvf4(tmem + C::kS, ad, bd, idS, tmem + C::kSFQ + 4 * kk, sfk + 4 * (kk >> 1) + 2 * (kk & 1), kk > 0);
        }
        mma_commit(s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      uint32_t pv_issued = 0;
      for (int i = 0; ok && i < n; ++i) {
        if (i + 1 < n && !(ok = issue_s(i + 1))) break;
        if (!(ok = mbar_wait(p_full(i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t pdesc_addr = sbase + C::kPOff + 4096 * (i & 1);
        const uint32_t sfp = tmem + C::kSFP + 4 * (i & 1);
        mma_nvf4(tmem + C::kL, smem_desc(pdesc_addr, 128, 256, 0), smem_desc(sbase + C::kOnesOff, 128, 256, 0), idL,
                 sfp, tmem + C::kSFO, 0);
        mma_commit(l_full);
        if (!(ok = mbar_wait(dec(i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t hot = gbits[i & 1][0] | gbits[i & 1][1] | gbits[i & 1][2] | gbits[i & 1][3];
        if (hot) list[count++] = (uint32_t)tile_of(i) | (hot << 16);
        if ((hot | invalid_groups) != 0xFFu) {
          const uint32_t blob = sbase + C::kStageOff + (i % C::NS) * C::kBlob;
          mma_nvf4(tmem + C::kO, smem_desc(pdesc_addr, 128, 256, 0), smem_desc(blob + blob_vcodes(D), 128, 256, 0),
                   idO, sfp, tmem + C::kSFV + 4 * sf_chunks(D) * (i & 1), pv_issued > 0);
          ++pv_issued;
        }
        mma_commit(pv_done(i & 1));
        mma_commit(blob_empty(i % C::NS));
      }
      p.hot_count[(size_t)bh * nblk + blk] = count;
      mma_commit(drain);
      wait_bounded(drain, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ one thread per row
    const int r = threadIdx.x, P = p0 + r;
    const bool valid = P < R;
    const int pos = valid ? P / G : 0;
    const int hq = h * G + (valid ? P % G : 0);
    const float cs = p.s_q[b * s.Hq + hq] * p.s_k[bh] * (kLog2e * rsqrtf((float)D));
    const int vis_last = s.causal ? pos + off : s.Nkv - 1;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float eps = p.eps;
    const bool eps_inf = isinf(eps);
    float m = -INFINITY, lam = 0.f, l = 0.f;
    bool ok = true;
    const int ngroups = s.ngroups(), nwords = (T + 31) / 32;
    for (int i = 0; i < n; ++i) {
      const int t = tile_of(i), j0 = t * kTile;
      const int nvis = valid ? min(kTile, vis_last + 1 - j0) : 0;
      if (!(ok = warp_wait(s_full, i & 1))) break;
      tc_fence_after();
      uint32_t sraw[64];
      tmem_ld_x32(tmem + lane_base + C::kS, sraw);
      tmem_ld_x32(tmem + lane_base + C::kS + 32, sraw + 32);
      tmem_wait_ld();
      float raw[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) raw[j] = __uint_as_float(sraw[j]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      if (nvis < kTile) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j >= nvis) raw[j] = -INFINITY;
      }
      float g[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = raw[16 * k];
#pragma unroll
        for (int j = 1; j < 15; j += 2) a = max3(a, raw[16 * k + j], raw[16 * k + j + 1]);
        g[k] = fmaxf(a, raw[16 * k + 15]);
      }
      const float c = fmaxf(fmaxf(g[0], g[1]), fmaxf(g[2], g[3])) * cs;  // tile max, log2 units
      const bool empty = (c == -INFINITY);
      const float mt = (c > m + kTau) ? c : m;  // candidate frame (lazy maximum)
      uint32_t pw[8];
      uint32_t sfw = 0x08080808u;  // 2^-6 where nothing is visible
      if (!empty) {
        sfw = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t sc = cvt_ue4m3(ex2_approx(fmaf(g[k], cs, -mt)) * (1.f / 6.f));
          sc = max(sc, 8u);  // clamp the group scale at 2^-6
          sfw |= sc << (8 * k);
          const float bias = mt + lg2_approx(ue4m3_value(sc));
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            uint32_t word = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 16 * k + 8 * w + 2 * e;
              const float a0 = ex2_approx(fmaf(raw[j], cs, -bias));
              const float a1 = ex2_approx(fmaf(raw[j + 1], cs, -bias));
              word |= cvt_e2m1x2(a0, a1) << (8 * e);
            }
            pw[2 * k + w] = word;
          }
        }
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) pw[w] = 0u;
      }
      // P buffer (and its scales) of this parity are free once PV(i-2) has completed
      if (i >= 2 && !(ok = warp_wait(pv_done(i & 1), ((i >> 1) - 1) & 1))) break;
      uint8_t* pb = smem + C::kPOff + 4096 * (i & 1) + (r >> 3) * 256 + (r & 7) * 16;
      *reinterpret_cast<uint4*>(pb) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(pb + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      const uint32_t sfp = tmem + lane_base + C::kSFP + 4 * (i & 1);
      tmem_st_x4(sfp, sfw, sfw, sfw, sfw);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(i & 1));
      // row sum of the quantized P (ones-MMA)
      if (!(ok = warp_wait(l_full, i & 1))) break;
      tc_fence_after();
      uint32_t lb;
      tmem_ld_x1(tmem + lane_base + C::kL, lb);
      tmem_wait_ld();
      const float ell = __uint_as_float(lb);
      // hot test: the group is hot if any of its rows exceeds eps * lambda
      bool vote = false;
      if (valid && !empty && !eps_inf) vote = (m == -INFINITY) ? (ell > 0.f) : (ell * ex2_approx(mt - m) > eps * lam);
      const uint32_t bal = __ballot_sync(0xffffffffu, vote);
      const bool hot_lo = (bal & 0x0000FFFFu) != 0, hot_hi = (bal & 0xFFFF0000u) != 0;
      const bool hot = lane < 16 ? hot_lo : hot_hi;
      bool rescale = false;
      float f = 1.f;
      if (!empty) {
        const float l_before = l;
        float mn;
        if (hot) {
          mn = fmaxf(m, c - kColdOffset);
          f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
          lam = lam * f + ell * ex2_approx(mt - mn);
          l *= f;
        } else {
          mn = mt;
          f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
          lam = lam * f + ell;
          l = l * f + ell;
        }
        rescale = (f != 1.f) && (l_before > 0.f);
        m = mn;
      }
      if (__any_sync(0xffffffffu, hot)) tmem_st_x4(sfp, hot ? 0u : sfw, hot ? 0u : sfw, hot ? 0u : sfw, hot ? 0u : sfw);
      if (__any_sync(0xffffffffu, rescale)) {
        if (!(ok = warp_wait(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1))) break;
        tc_fence_after();
        const float fr = rescale ? f : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tmem + lane_base + C::kO + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * fr);
          tmem_st_x16(tmem + lane_base + C::kO + c0, o);
          tmem_st_x16(tmem + lane_base + C::kO + c0 + 16, o + 16);
        }
      }
      if (lane == 0) gbits[i & 1][warp] = ((uint32_t)hot_lo << (2 * warp)) | ((uint32_t)hot_hi << (2 * warp + 1));
      if (p.hot_mask && (lane == 0 || lane == 16) && hot) {
        const int grp = (p0 + 32 * warp + lane) / kGroupRows;
        if (grp < ngroups) atomicOr(&p.hot_mask[((size_t)bh * ngroups + grp) * nwords + t / 32], 1u << (t % 32));
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dec(i & 1));
    }
    // ---- epilogue: write the pass-1 state (o scaled by s_v, frame m, cold sum l)
    if (ok && n > 0) ok = warp_wait(pv_done((n - 1) & 1), ((n - 1) >> 1) & 1);
    tc_fence_after();
    if (ok) {
      const float sv = p.s_v[bh];
      float* orow = p.state_o + ((size_t)bh * nblk * kBlockRows + P) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld_x32(tmem + lane_base + C::kO + c0, o);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(orow + c0 + j) =
              l > 0.f ? make_float4(__uint_as_float(o[j]) * sv, __uint_as_float(o[j + 1]) * sv,
                                    __uint_as_float(o[j + 2]) * sv, __uint_as_float(o[j + 3]) * sv)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      p.state_ml[(size_t)bh * nblk * kBlockRows + P] = make_float2(m, l);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const P1Params& prm, cudaStream_t st) {
  const int smem = P1Cfg<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(pass1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  pass1_kernel<D><<<prm.s.BH() * prm.s.nblk(), kThreads, smem, st>>>(prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pass1(const Shape& s, const Workspace& ws, float eps, uint32_t* hot_mask, cudaStream_t st) {
  P1Params prm{};
  prm.s = s;
  prm.kv_blob = ws.kv_blob;
  prm.q_blob = ws.q_blob;
  prm.s_k = ws.s_k;
  prm.s_v = ws.s_v;
  prm.s_q = ws.s_q;
  prm.eps = eps;
  prm.state_o = ws.state_o;
  prm.state_ml = ws.state_ml;
  prm.hot_list = ws.hot_list;
  prm.hot_count = ws.hot_count;
  prm.hot_mask = hot_mask;
  prm.err = device_error_word();
  switch (s.d) {
    case 64: return launch_d<64>(prm, st);
    case 128: return launch_d<128>(prm, st);
    case 256: return launch_d<256>(prm, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace apa
