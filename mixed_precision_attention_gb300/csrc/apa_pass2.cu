// apa_pass2.cu -- exact BF16 attention over a list of key tiles, merged with
// the pass-1 state.
//
// "APA: sloppy attention, exact where it counts" (rfriedmann.de blog),
// "Pass 2: exact FP16 on the hot tiles": a pass-2 CTA takes the same rows as a
// pass-1 CTA, collects the union of their hot tiles, computes each row only on
// its own group's hot tiles with an FP32 online softmax, and merges with the
// pass-1 state ("The merge that makes it exact").  Logits are centred by the
// same per-channel key mean as pass 1 (q.k - q.mu), so both states share one
// frame; the natural-log LSE adds q.mu/sqrt(d) back.
//
// With eps = 0 the same kernels are the all-exact path: every visible tile of
// the block, no pass-1 state, uncentred logits.
//
// GB300 design: one CTA = one 128-row block of GQA-packed rows of one KV head
// (tcgen05 M = 128), 7 warps:
//   warps 0-3  softmax, one thread per row (TMEM lane = row);
//   warp 4     TMA producer: K and V tiles (64 keys x d, 128-byte swizzle) into an
//              NS-stage ring;
//   warp 5     TMEM owner and S issuer: S = Q K^T (kind::f16, K-major x K-major)
//              into a double-buffered S in TMEM;
//   warp 6     PV issuer: O += P V (V MN-major) into O in TMEM.
// A tcgen05.mma takes tens of cycles to issue, and one tile needs d/16 of them
// for S and 4 (or 8) for PV: issued by one thread, they set the tile period.
// The running max moves lazily (only when a score exceeds it by more than 8 in
// log2 units), so O in TMEM is rarely rescaled.  P goes to the tensor cores as
// one FP16 term (relative rounding error at most 2^-11) against an FP16 copy of
// V (V divided by a power of two per head, exact for every bf16 value above the
// FP16 subnormals), which the quantizer writes in APA mode and a conversion
// pass writes in the all-exact mode.
// K may come from a paged pool through a block table: its tensor map then spans
// the pool, and the rows past Nkv of the last page are zeroed in shared memory
// before any MMA reads them.
//
// At d <= 128 a second kernel (pass2_dual_kernel) runs instead: two
// softmax warp groups per block take alternate entries of the hot list, each
// with its own (m, l), its own O in TMEM and its own double-buffered S, so one
// group's exp/convert/store of P overlaps the other's S and PV MMAs.  13 warps:
// eight softmax, a TMA producer each for K (8-stage ring) and V (4 stages), an S
// issuer per group and one PV issuer.  P never goes through shared memory: each
// softmax thread writes its row of P (FP16) over the first half of the S slot it
// read, and the PV product takes its A operand from TMEM; an S issuer writes the
// next S into a slot only after the P.V that read the slot's P has completed.
// The block's final state is the merge of the pass-1 state, group 0's and group
// 1's, in that order.  The per-row work is
// the same as the one-group kernel's; only the tile-to-accumulator assignment
// (and so the rounding order of the merge) differs.
#include <cstring>
#include <cuda_fp16.h>

#include "apa_internal.h"
#include "tc.cuh"

namespace apa {

namespace {

struct P2Params {
  Shape s;
  const uint16_t* q;
  const float* mu;            // null in the all-exact mode
  const float* state_o;       // pass-1 o [BH][nblk*128][d] or null
  const float2* state_ml;     // pass-1 (m, l) [BH][nblk*128] or null
  const uint32_t* hot_list;   // [BH*nblk][T] or null (all visible tiles)
  const uint32_t* hot_count;  // [BH*nblk] or null
  const uint32_t* order;      // [BH*nblk] work items, longest hot list first, or null
  const uint32_t* vamax;      // [BH] max |v| (float bits): the FP16 V copy's scale, or null
  float* out;                 // [B,Hq,Nq,d]
  float* lse;                 // [B,Hq,Nq] or null
  int* err;
  // the one-group kernel (d = 256) can split each block's walk (all visible tiles, or
  // the hot list) into nsplit parts, one CTA each, which write their states (O in the
  // FP16-V copy's units, and (m, l)) at row (item * nsplit + part) * 128 + r, item =
  // bh * nblk + blk, for combine_kernel to merge.  In APA mode part 0 also carries
  // the pass-1 state, and writes each row's LSE term q.mu / sqrt(d).
  int nsplit;
  float* part_o;              // [BH*nblk*nsplit][128][d]
  float2* part_ml;            // [BH*nblk*nsplit][128]
  float* part_qmu;            // [BH*nblk][128], APA mode only
};

constexpr int kThreads = 224;
#ifndef APA_P2_STAGES_D128
#define APA_P2_STAGES_D128 4  // K/V stages of the FP16 pass 2 at d = 128
#endif
constexpr float kTau2 = 8.0f;  // pass-2 lazy rescale threshold (log2 units)

// The barriers live at the end of the dynamic shared-memory window and there is
// no static shared memory.  With kCtasPerSm = 2 (2 K/V stages, 112 KB per CTA at
// d = 128 when P still went through shared memory) two CTAs would fit an SM with
// no alignment slack; the kernel then checks that the window starts on a
// 1024-byte boundary (the 128-byte swizzle needs it).  Measured on the 2048 x
// 122880 layer, two CTAs of that shape were no faster than one CTA with 3 stages.
// P goes from the softmax threads into TMEM, over the S slot it came from, and the
// PV product reads it there.
template <int D>
struct P2Cfg {
  static constexpr int kCtasPerSm = 1;
  static constexpr int NS = kCtasPerSm == 2 ? 2 : (D >= 256 ? 2 : (D == 128 ? APA_P2_STAGES_D128 : 3));
  static constexpr int kAtoms = D / 64;
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kKVBytes = 64 * D * 2;  // one of K or V per stage
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQBytes;
  static constexpr int kNumBars = 2 * NS + 10;
  static constexpr int kBarOff = kStageOff + NS * 2 * kKVBytes;
  static constexpr int kSlack = kCtasPerSm == 2 ? 0 : 1024;  // runtime alignment room
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + kSlack;
  static constexpr uint32_t kTmemCols = D + 128 <= 256 ? 256 : 512;
  static constexpr uint32_t kOCol = 0, kSCol = D;
};

__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, int* err) {
  // used only while unwinding: waits for copies already in flight, ignoring the abort flag
  const unsigned long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > APA_WAIT_LIMIT_CYCLES) {
      if (err) atomicCAS(err, 0, APA_DEVERR_TIMEOUT);
      return;
    }
  }
}

// P of eight consecutive keys, 2^(x*c2 + nb), as four FP16x2 words (key 2k in the
// low half of word k); the FP32 values are added into (s0, s1): even keys into s0,
// odd keys into s1.  The affine step and the sums run as packed FP32 pairs.
__device__ __forceinline__ void p8_f16(const float* x, float c2, float nb, uint32_t* h, float& s0, float& s1) {
  asm("{\n.reg .b64 a0, a1, a2, a3, c, n, s, one;\n"
      ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n"
      "mov.b64 c, {%14, %14};\n"
      "mov.b64 n, {%15, %15};\n"
      "mov.b64 one, {%16, %16};\n"
      "mov.b64 a0, {%6, %7};\n"
      "mov.b64 a1, {%8, %9};\n"
      "mov.b64 a2, {%10, %11};\n"
      "mov.b64 a3, {%12, %13};\n"
      "fma.rn.f32x2 a0, a0, c, n;\n"
      "fma.rn.f32x2 a1, a1, c, n;\n"
      "fma.rn.f32x2 a2, a2, c, n;\n"
      "fma.rn.f32x2 a3, a3, c, n;\n"
      "mov.b64 {y0, y1}, a0;\n"
      "mov.b64 {y2, y3}, a1;\n"
      "mov.b64 {y4, y5}, a2;\n"
      "mov.b64 {y6, y7}, a3;\n"
      "ex2.approx.ftz.f32 y0, y0;\n"
      "ex2.approx.ftz.f32 y1, y1;\n"
      "ex2.approx.ftz.f32 y2, y2;\n"
      "ex2.approx.ftz.f32 y3, y3;\n"
      "ex2.approx.ftz.f32 y4, y4;\n"
      "ex2.approx.ftz.f32 y5, y5;\n"
      "ex2.approx.ftz.f32 y6, y6;\n"
      "ex2.approx.ftz.f32 y7, y7;\n"
      "cvt.rn.f16x2.f32 %0, y1, y0;\n"
      "cvt.rn.f16x2.f32 %1, y3, y2;\n"
      "cvt.rn.f16x2.f32 %2, y5, y4;\n"
      "cvt.rn.f16x2.f32 %3, y7, y6;\n"
      "mov.b64 s, {%4, %5};\n"
      "mov.b64 a0, {y0, y1};\n"
      "mov.b64 a1, {y2, y3};\n"
      "mov.b64 a2, {y4, y5};\n"
      "mov.b64 a3, {y6, y7};\n"
      "fma.rn.f32x2 s, a0, one, s;\n"
      "fma.rn.f32x2 s, a1, one, s;\n"
      "fma.rn.f32x2 s, a2, one, s;\n"
      "fma.rn.f32x2 s, a3, one, s;\n"
      "mov.b64 {%4, %5}, s;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]), "+f"(s0), "+f"(s1)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]), "f"(c2), "f"(nb),
        "f"(1.f));
}

template <int D>
__global__ void __launch_bounds__(kThreads, P2Cfg<D>::kCtasPerSm)
    pass2_kernel(const P2Params p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using C = P2Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (C::kSlack == 0 && smem != smem_raw) {  // no room to realign: refuse loudly
    if (threadIdx.x == 0) atomicCAS(p.err, 0, APA_DEVERR_SMEM_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  int& abort_flag = *reinterpret_cast<int*>(smem + C::kBarOff + C::kNumBars * 8 + 4);

  const Shape& s = p.s;
  const int nblk = s.nblk(), BH = s.BH(), G = s.G(), R = s.R(), T = s.T(), off = s.off();
  // longest hot lists first when ranked, else heavy (late, causal) blocks first:
  // CTAs start in index order, so the longest work items start earliest
  int bh, blk;
  const int part = p.nsplit > 1 ? (int)blockIdx.x % p.nsplit : 0;
  const int cta = p.nsplit > 1 ? (int)blockIdx.x / p.nsplit : (int)blockIdx.x;
  if (p.order) {
    const int item = (int)p.order[cta];
    bh = item / nblk;
    blk = item % nblk;
  } else {
    bh = cta % BH;
    blk = nblk - 1 - cta / BH;
  }
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  const int p0 = blk * kBlockRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto kv_full = [&](int st) { return bar0 + 8u * st; };
  auto kv_empty = [&](int st) { return bar0 + 8u * (C::NS + st); };
  auto s_full = [&](int b2) { return bar0 + 8u * (2 * C::NS + b2); };
  // (slots 2 NS + 2, 3 are unused: an S slot is free once the P.V that reads the P
  // written over it has completed, so pv_done tells the S issuer)
  auto p_full = [&](int b2) { return bar0 + 8u * (2 * C::NS + 4 + b2); };
  auto pv_done = [&](int b2) { return bar0 + 8u * (2 * C::NS + 6 + b2); };
  const uint32_t drain = bar0 + 8u * (2 * C::NS + 8), drain_pv = bar0 + 8u * (2 * C::NS + 9);
  // every lane of a softmax warp waits; the warp proceeds only if all lanes succeeded
  auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;  // already complete
    const bool okl = mbar_wait(bar, parity, &abort_flag, p.err);
    return __all_sync(0xffffffffu, okl);
  };

  // the block's tile list; with a split walk this CTA's part of it
  const bool apa_mode = p.hot_list != nullptr;
  const int last_row = min(R, p0 + kBlockRows) - 1;
  const int t_hi = s.causal ? min(T - 1, (last_row / G + off) / kTile) : T - 1;
  const int n_all = apa_mode ? (int)p.hot_count[(size_t)bh * nblk + blk] : t_hi + 1;
  const int i0 = p.nsplit > 1 ? (int)((long long)n_all * part / p.nsplit) : 0;
  const int n = p.nsplit > 1 ? (int)((long long)n_all * (part + 1) / p.nsplit) - i0 : n_all;
  const uint32_t* list = apa_mode ? p.hot_list + ((size_t)bh * nblk + blk) * T : nullptr;
  auto tile_of = [&](int i, uint32_t& gmask) -> int {
    if (apa_mode) {
      const uint32_t e = list[i0 + i];
      gmask = e >> 16;
      return (int)(e & 0xFFFFu);
    }
    gmask = 0xFFu;
    const int g = i0 + i;
    return g == 0 ? 0 : t_hi + 1 - g;
  };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::kNumBars; ++i) {
      const bool per_warp = (i >= 2 * C::NS + 4 && i < 2 * C::NS + 6);  // p_full: one arrive per softmax warp
      const bool kv_empty_bar = (i >= C::NS && i < 2 * C::NS);           // kv_empty: the S and the PV issuer
      mbar_init(bar0 + 8u * i, per_warp ? 4u : (kv_empty_bar ? 2u : 1u));
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }

  // ---- softmax-thread setup: Q row into smem (128-byte swizzle, K-major), q.mu
  const int r = threadIdx.x;  // row within the block for warps 0-3
  const int P = p0 + r;
  const bool row_valid = warp < 4 && P < R;
  const int pos = row_valid ? P / G : 0;
  const int hq = h * G + (row_valid ? P % G : 0);
  float qmu = 0.f;
  if (warp < 4) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (((size_t)b * s.Hq + hq) * s.Nq + pos) * D);
    const float* mu = p.mu ? p.mu + (size_t)bh * D : nullptr;
#pragma unroll 4
    for (int j = 0; j < D / 8; ++j) {
      uint4 val = row_valid ? src[j] : make_uint4(0u, 0u, 0u, 0u);
      const int atom = j >> 3, chunk = j & 7;
      *reinterpret_cast<uint4*>(smem + C::kQOff + atom * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4)) = val;
      if (mu) {
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qmu = fmaf(__uint_as_float(w[e] << 16), mu[j * 8 + 2 * e], qmu);
          qmu = fmaf(__uint_as_float(w[e] & 0xFFFF0000u), mu[j * 8 + 2 * e + 1], qmu);
        }
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(kv_empty(st), ((i / C::NS) - 1) & 1, &abort_flag, p.err)) break;
        uint32_t gm;
        const int t = tile_of(i, gm);
        // contiguous maps: (channel, key, b * Hkv + h); paged maps: (channel, key in
        // page, page * Hkv + h).  The FP16 copy of V is contiguous in either case.
        int ky = t * kTile, kz = bh;
        const int vy = ky, vz = bh;
        if (s.pages) {
          ky = 0;
          kz = kv_page(s, b, t, p.err) * s.Hkv + h;
        }
        mbar_arrive_expect_tx(kv_full(st), 2 * C::kKVBytes);
        const uint32_t kdst = sbase + C::kStageOff + st * 2 * C::kKVBytes;
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) {
          tma_load_3d(kdst + a * 8192, &kmap, a * 64, ky, kz, kv_full(st));
          tma_load_3d(kdst + C::kKVBytes + a * 8192, &vmap, a * 64, vy, vz, kv_full(st));
        }
        issued = i + 1;
      }
      // every copy issued lands before the CTA exits, also when another warp gave up
      // after this loop ended (normally they have all landed: the waits return at once)
      for (int i = max(0, issued - C::NS); i < issued; ++i) wait_bounded(kv_full(i % C::NS), (i / C::NS) & 1, p.err);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0 && n > 0) {
      const uint32_t idS = idesc_bf16(128, 64, 0);
      auto issue_s = [&](int i) -> bool {
        const int st = i % C::NS;
        if (!mbar_wait(kv_full(st), (i / C::NS) & 1, &abort_flag, p.err)) return false;
        uint32_t gm_unused;
        if (s.pages && (s.Nkv % kTile) != 0 && tile_of(i, gm_unused) == T - 1) {
          // paged pool: the keys past Nkv in a sequence's last page hold whatever the
          // pool holds there (possibly NaN or Inf).  Masked scores and a zero P do not
          // keep those out of an MMA, so the K rows are zeroed here, before any MMA
          // reads this stage (V comes from the contiguous FP16 copy).
          const int nk = s.Nkv - (T - 1) * kTile, rows = kTile - nk;
          uint8_t* kst = smem + C::kStageOff + st * 2 * C::kKVBytes;
          for (int x = 0; x < rows * C::kAtoms * 8; ++x) {
            const int rest = x >> 3, rr = nk + rest % rows, atom = rest / rows;
            *reinterpret_cast<uint4*>(kst + atom * 8192 + rr * 128 + (x & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // the slot holds P of entry i - 2 until its P.V has read it
        if (i >= 2 && !mbar_wait(pv_done(i & 1), ((i >> 1) - 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t kaddr = sbase + C::kStageOff + st * 2 * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc(sbase + C::kQOff + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(kaddr + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          mma_bf16(tmem + C::kSCol + 64 * (i & 1), ad, bd, idS, kk > 0);
        }
        mma_commit(s_full(i & 1));
        mma_commit(kv_empty(st));  // this stage's K has been read
        return true;
      };
      for (int i = 0; i < n; ++i)
        if (!issue_s(i)) break;
      // drain: every tcgen05 op issued by this thread has completed before TMEM is freed
      mma_commit(drain);
      wait_bounded(drain, 0, p.err);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0 && n > 0) {
      const uint32_t idO = idesc_f16(128, D, 1);
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        if (!(ok = mbar_wait(p_full(i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
        if (!(ok = mbar_wait(kv_full(i % C::NS), (i / C::NS) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t vaddr = sbase + C::kStageOff + (i % C::NS) * 2 * C::kKVBytes + C::kKVBytes;
        // P (FP16) sits in the first 32 columns of its S slot: 16 keys per MMA
        const uint32_t pcol = tmem + C::kSCol + 64u * (i & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = smem_desc(vaddr + kk * 2048, 8192, 1024, kSwizzle128B);
          mma_f16_ts(tmem + C::kOCol, pcol + 8u * kk, bd, idO, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(pv_done(i & 1));
        mma_commit(kv_empty(i % C::NS));  // this stage's V has been read
      }
      mma_commit(drain_pv);
      wait_bounded(drain_pv, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax (one thread per row)
    const float c2 = kLog2e * rsqrtf((float)D);
    const float shift = p.mu ? qmu * c2 : 0.f;
    const int vis_last = s.causal ? pos + off : s.Nkv - 1;  // last visible key of this row
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m2 = -INFINITY, l2 = 0.f;
    bool ok = true;
    // the hot-list entry of the next tile is loaded one tile ahead, off the critical path
    uint32_t gm_next = 0;
    int t_next = n > 0 ? tile_of(0, gm_next) : 0;
    for (int i = 0; i < n; ++i) {
      const uint32_t gm = gm_next;
      const int t = t_next;
      if (i + 1 < n) t_next = tile_of(i + 1, gm_next);
      if (!(ok = warp_wait(s_full(i & 1), (i >> 1) & 1))) break;
      const bool row_hot = row_valid && ((gm >> (r >> 4)) & 1u);
      const int j0 = t * kTile;
      const int nvis = row_hot ? min(kTile, vis_last + 1 - j0) : 0;  // keys j0 .. j0+nvis-1 visible
      // P (FP16, two keys per column) goes over the first 32 columns of the S slot it
      // came from; the slot's previous P had been read before S was written into it
      const uint32_t pslot = tmem + lane_base + C::kSCol + 64u * (i & 1);
      tc_fence_after();
      if (!__any_sync(0xffffffffu, nvis > 0)) {
        // neither of this warp's two groups takes part in this tile: its P rows are zero
        uint32_t z[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) z[x] = 0u;
        tmem_st_x16(pslot, z);
        tmem_st_x16(pslot + 16, z);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(i & 1));
        continue;
      }
      uint32_t raw[64];
      tmem_ld_x32(pslot, raw);
      tmem_ld_x32(pslot + 32, raw + 32);
      tmem_wait_ld();
      // raw scores.  Keys past a row's last visible one are masked to -inf only on
      // the diagonal (0 < nvis < 64); a row with nothing visible here (cold group or
      // beyond the diagonal) keeps its scores but takes no part: its maximum is -inf
      // and its P bias -inf, so its P is exactly 0.
      float sv[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) sv[j] = __uint_as_float(raw[j]);
      if (__any_sync(0xffffffffu, nvis > 0 && nvis < 64)) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j >= nvis) sv[j] = -INFINITY;
      }
      // row maximum as a tree of 3-input maxima; the logit map x*c2 - shift is monotone
      // (c2 > 0), so its maximum is the map of the raw maximum, rounded the same way
      float g8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        g8[k] = max3(max3(sv[8 * k], sv[8 * k + 1], sv[8 * k + 2]), max3(sv[8 * k + 3], sv[8 * k + 4], sv[8 * k + 5]),
                     fmaxf(sv[8 * k + 6], sv[8 * k + 7]));
      const float rmax = max3(max3(g8[0], g8[1], g8[2]), max3(g8[3], g8[4], g8[5]), fmaxf(g8[6], g8[7]));
      const float c = (nvis <= 0 || rmax == -INFINITY) ? -INFINITY : fmaf(rmax, c2, -shift);
      float f = 1.f;
      bool rescale = false;
      if (c > m2 + kTau2 || (m2 == -INFINITY && c > -INFINITY)) {
        if (l2 > 0.f) {
          f = ex2_approx(m2 - c);
          rescale = true;
        }
        m2 = c;
      }
      // P = 2^(x*c2 - shift - m2), one bias per row; -inf for a row with nothing
      // visible in this tile (finite scores times c2 plus -inf give 2^-inf = 0)
      const float nb = (nvis <= 0 || m2 == -INFINITY) ? -INFINITY : -shift - m2;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};  // four partial row sums (short dependency chains)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // the row sum adds the FP32 values; their FP16 roundings (relative error
        // at most 2^-11 each) go to the tensor cores
        uint32_t pk[16];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int ch = 4 * hf + c4;
          p8_f16(sv + 8 * ch, c2, nb, pk + 4 * c4, ps[ch & 1], ps[2 + (ch & 1)]);
        }
        tmem_st_x16(pslot + 16u * hf, pk);
      }
      l2 = l2 * f + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      if (__any_sync(0xffffffffu, rescale)) {
        // O must not be read before PV(i-1) has landed
        if (!(ok = warp_wait(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tmem + lane_base + C::kOCol + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
          tmem_st_x16(tmem + lane_base + C::kOCol + c0, o);
          tmem_st_x16(tmem + lane_base + C::kOCol + c0 + 16, o + 16);
        }
      }
      tmem_wait_st();  // P (and a rescaled O) in TMEM before P.V is issued
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(i & 1));
    }
    // ---- epilogue: merge with the pass-1 state, write out and lse (or, for one part
    // of a split walk, this part's state)
    if (ok && n > 0) ok = warp_wait(pv_done((n - 1) & 1), ((n - 1) >> 1) & 1);
    tc_fence_after();
    if (ok && p.nsplit > 1) {
      const size_t item = (size_t)bh * nblk + blk;
      const size_t prow = (item * p.nsplit + part) * kBlockRows + r;
      float* po = p.part_o + prow * D;
      // APA mode, part 0: the pass-1 state merged in first (as the epilogue below
      // does), in the FP16-V copy's units (a division by a power of two)
      float w1 = 0.f, w2 = 1.f, mo = m2, lo = l2, inv_vsc = 1.f;
      const float* st = nullptr;
      if (part == 0 && p.state_o) {
        float m1 = -INFINITY, l1 = 0.f;
        st = p.state_o + ((size_t)bh * nblk * kBlockRows + P) * D;
        if (row_valid) {
          const float2 ml = p.state_ml[(size_t)bh * nblk * kBlockRows + P];
          m1 = ml.x;
          l1 = ml.y;
        }
        const float e1 = l1 > 0.f ? m1 : -INFINITY, e2 = l2 > 0.f ? m2 : -INFINITY;
        mo = fmaxf(e1, e2);
        w1 = e1 == -INFINITY ? 0.f : exp2f(e1 - mo);
        w2 = e2 == -INFINITY ? 0.f : exp2f(e2 - mo);
        lo = w1 * l1 + w2 * l2;
        inv_vsc = 1.f / v16_scale(__uint_as_float(p.vamax[bh]));
        if (p.mu) p.part_qmu[item * kBlockRows + r] = qmu * rsqrtf((float)D);
      }
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld_x32(tmem + lane_base + C::kOCol + c0, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        if (st && row_valid) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            o[j] = __float_as_uint(w1 * (st[c0 + j] * inv_vsc) + w2 * __uint_as_float(o[j]));
        }
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(po + c0 + j) = make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]),
                                                                __uint_as_float(o[j + 2]), __uint_as_float(o[j + 3]));
      }
      p.part_ml[prow] = make_float2(mo, lo);
    } else if (ok) {
      float m1 = -INFINITY, l1 = 0.f;
      const float* st = nullptr;
      if (p.state_o) {
        st = p.state_o + ((size_t)bh * nblk * kBlockRows + P) * D;
        if (row_valid) {
          const float2 ml = p.state_ml[(size_t)bh * nblk * kBlockRows + P];
          m1 = ml.x;
          l1 = ml.y;
        }
      }
      const float e1 = l1 > 0.f ? m1 : -INFINITY, e2 = l2 > 0.f ? m2 : -INFINITY;
      const float M = fmaxf(e1, e2);
      const float w1 = e1 == -INFINITY ? 0.f : exp2f(e1 - M), w2 = e2 == -INFINITY ? 0.f : exp2f(e2 - M);
      const float L = w1 * l1 + w2 * l2;
      const float invL = 1.f / L;
      const float w2o = w2 * v16_scale(__uint_as_float(p.vamax[bh]));  // O carries V / scale
      float* orow = p.out + (((size_t)b * s.Hq + hq) * s.Nq + pos) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld_x32(tmem + lane_base + C::kOCol + c0, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float4 res;
            float* rr = &res.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a1 = st ? st[c0 + j + e] : 0.f;
              rr[e] = (w1 * a1 + w2o * __uint_as_float(o[j + e])) * invL;
            }
            *reinterpret_cast<float4*>(orow + c0 + j) = res;
          }
        }
      }
      if (row_valid && p.lse) {
        const float lg = M + log2f(L);
        p.lse[((size_t)b * s.Hq + hq) * s.Nq + pos] = 0.6931471805599453f * lg + (p.mu ? qmu * rsqrtf((float)D) : 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Barrier over the two softmax warp groups (named barrier 1, 256 threads), also
// returning whether v held in all of them.
__device__ __forceinline__ bool dual_sync_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.and.pred q, 1, 256, p;\n"
      "selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// ----------------------------------------------------------------------------
// Pass 2 in APA mode (FP16 P.V, d <= 128) with two softmax warp groups on one
// 128-row block: group u takes the hot-list entries i with i % 2 == u, with its
// own online softmax (m, l) and its own O accumulator in TMEM, so the two
// groups' per-tile latencies overlap.  At the end the pass-1 state and the two
// groups' states are merged, always in that order.  TMEM: two O accumulators and
// a double-buffered S per group (512 columns).
//
// K and V travel in rings of their own, each filled by its own TMA warp: S(i)
// then waits only for the K ring to free a stage (S(i - NSK) done), not for the
// P.V product of an older tile, so the S MMAs run up to NSK tiles ahead.  Each
// group has its own S-issuing warp; the PV warp serves both groups in list order.
#ifndef APA_P2D_KSTAGES
#define APA_P2D_KSTAGES 8  // K stages of the two-group pass 2 (even: see P2DualCfg)
#endif
#ifndef APA_P2D_VSTAGES
#define APA_P2D_VSTAGES 4  // V stages of the two-group pass 2
#endif
template <int D>
struct P2DualCfg {
  static constexpr int NS = APA_P2D_KSTAGES;   // K stages
  static constexpr int NSV = APA_P2D_VSTAGES;  // V stages
  static constexpr int kAtoms = D / 64;
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kKVBytes = 64 * D * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + NS * kKVBytes;
  // (P goes from the softmax threads into TMEM, over the S slot it came from)
  static constexpr int kMlOff = kVOff + NSV * kKVBytes;  // group 1's (m, l) per row for the merge
  static constexpr int kSIssuers = 2;  // S-issuing warps: one per group
  // The two S issuers each wait on the K arrivals of their own entries (i % 2).  With
  // NS even, entry i's K stage i % NS is only ever used by entries of the same
  // parity, so each issuer sees every phase of its stages in order.  With NS odd, a
  // stage's previous use would be the other issuer's; a parity wait made one phase
  // early (the previous load still landing, since loads can land out of order) would
  // pass on the phase before it.
  static_assert(NS % 2 == 0, "two S issuers need an even K stage count");
  static constexpr int kB0 = 2 * NS + 2 * NSV;
  static constexpr int kNumBars = kB0 + 16 + 1 + kSIssuers;
  static constexpr int kBarOff = kMlOff + 128 * 8;
  static constexpr int kSmem = kBarOff + kNumBars * 8 + 16 + 1024;
  static_assert(kSmem <= 232448, "shared memory");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSBase = 2 * D;  // S(u, b) at kSBase + 128 u + 64 b; O(u) at D u
  static constexpr int kThreads = 13 * 32;
  static_assert(kSBase + 256 <= kTmemCols, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(P2DualCfg<D>::kThreads, 1)
    pass2_dual_kernel(const P2Params p, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using C = P2DualCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  int& abort_flag = *reinterpret_cast<int*>(smem + C::kBarOff + C::kNumBars * 8 + 4);
  float2* ml1 = reinterpret_cast<float2*>(smem + C::kMlOff);

  const Shape& s = p.s;
  const int nblk = s.nblk(), BH = s.BH(), G = s.G(), R = s.R(), T = s.T(), off = s.off();
  int bh, blk;
  if (p.order) {
    const int item = (int)p.order[blockIdx.x];
    bh = item / nblk;
    blk = item % nblk;
  } else {
    bh = blockIdx.x % BH;
    blk = nblk - 1 - (int)(blockIdx.x / BH);
  }
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  const int p0 = blk * kBlockRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // warps 0-7 softmax, 8 TMA producer of K, 9 S issuer of group 0's tiles, 10 PV
  // issuer, 11 S issuer of group 1's tiles, 12 TMA producer of V
  const int kProd = 8, kMmaS = 9, kMmaPV = 10, kMmaS1 = 11, kProdV = 12;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto k_full = [&](int st) { return bar0 + 8u * st; };
  auto k_empty = [&](int st) { return bar0 + 8u * (C::NS + st); };
  auto v_full = [&](int st) { return bar0 + 8u * (2 * C::NS + st); };
  auto v_empty = [&](int st) { return bar0 + 8u * (2 * C::NS + C::NSV + st); };
  auto s_full = [&](int u, int b2) { return bar0 + 8u * (C::kB0 + 8 * u + b2); };
  // (slots kB0 + 8 u + 2, 3 are unused: a slot of S is free once the P.V that reads
  // the P written over it has completed, so pv_done tells the S issuers)
  auto p_full = [&](int u, int b2) { return bar0 + 8u * (C::kB0 + 8 * u + 4 + b2); };
  auto pv_done = [&](int u, int b2) { return bar0 + 8u * (C::kB0 + 8 * u + 6 + b2); };
  const uint32_t drain_pv = bar0 + 8u * (C::kB0 + 16);
  auto drain_s = [&](int x) { return bar0 + 8u * (C::kB0 + 17 + x); };  // per S issuer
  auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    const bool okl = mbar_wait(bar, parity, &abort_flag, p.err);
    return __all_sync(0xffffffffu, okl);
  };

  // the block's tiles: its hot list (APA mode), or every tile it sees in the order
  // 0, t_hi, ..., 1 with all eight row groups taking part (all-exact mode)
  const bool apa_mode = p.hot_list != nullptr;
  const int last_row = min(R, p0 + kBlockRows) - 1;
  const int t_hi = s.causal ? min(T - 1, (last_row / G + off) / kTile) : T - 1;
  const int n = apa_mode ? (int)p.hot_count[(size_t)bh * nblk + blk] : t_hi + 1;
  const uint32_t* list = apa_mode ? p.hot_list + ((size_t)bh * nblk + blk) * T : nullptr;
  auto entry = [&](int i) -> uint32_t {
    return apa_mode ? list[i] : ((uint32_t)(i == 0 ? 0 : t_hi + 1 - i) | (0xFFu << 16));
  };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::kNumBars; ++i) {
      uint32_t count = 1;
      const int j = i - C::kB0;
      if (j >= 0 && j < 16 && (j & 7) >= 4 && (j & 7) < 6) count = 4;  // p_full: the group's four warps
      mbar_init(bar0 + 8u * i, count);
    }
    fence_mbar_init();
  }
  if (warp == kMmaS) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProd && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }

  // ---- softmax-thread setup: the Q row (group 0 stores it, 128-byte swizzle), q.mu (both groups)
  const int u = warp >> 2, qw = warp & 3;  // softmax warps 0-7: group u, quarter qw
  const int r = qw * 32 + lane;            // row within the block
  const int P = p0 + r;
  const bool row_valid = warp < 8 && P < R;
  const int pos = row_valid ? P / G : 0;
  const int hq = h * G + (row_valid ? P % G : 0);
  float qmu = 0.f;
  if (warp < 8) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (((size_t)b * s.Hq + hq) * s.Nq + pos) * D);
    const float* mu = p.mu ? p.mu + (size_t)bh * D : nullptr;  // null: uncentred logits
#pragma unroll 4
    for (int j = 0; j < D / 8; ++j) {
      uint4 val = row_valid ? src[j] : make_uint4(0u, 0u, 0u, 0u);
      const int atom = j >> 3, chunk = j & 7;
      if (u == 0)
        *reinterpret_cast<uint4*>(smem + C::kQOff + atom * 16384 + r * 128 + ((chunk ^ (r & 7)) << 4)) = val;
      if (mu) {
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qmu = fmaf(__uint_as_float(w[e] << 16), mu[j * 8 + 2 * e], qmu);
          qmu = fmaf(__uint_as_float(w[e] & 0xFFFF0000u), mu[j * 8 + 2 * e + 1], qmu);
        }
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kProd) {
    // ------------------------------------------------------------ TMA producer of K
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(k_empty(st), ((i / C::NS) - 1) & 1, &abort_flag, p.err)) break;
        const int t = (int)(entry(i) & 0xFFFFu);
        int ky = t * kTile, kz = bh;
        if (s.pages) {
          ky = 0;
          kz = kv_page(s, b, t, p.err) * s.Hkv + h;
        }
        mbar_arrive_expect_tx(k_full(st), C::kKVBytes);
        const uint32_t kdst = sbase + C::kKOff + st * C::kKVBytes;
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) tma_load_3d(kdst + a * 8192, &kmap, a * 64, ky, kz, k_full(st));
        issued = i + 1;
      }
      // every copy issued lands before the CTA exits, also when another warp gave up
      // after this loop ended (normally they have all landed: the waits return at once)
      for (int i = max(0, issued - C::NS); i < issued; ++i) wait_bounded(k_full(i % C::NS), (i / C::NS) & 1, p.err);
    }
  } else if (warp == kProdV) {
    // ------------------------------------------------------------ TMA producer of V
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NSV;
        if (i >= C::NSV && !mbar_wait(v_empty(st), ((i / C::NSV) - 1) & 1, &abort_flag, p.err)) break;
        const int t = (int)(entry(i) & 0xFFFFu);
        mbar_arrive_expect_tx(v_full(st), C::kKVBytes);
        const uint32_t vdst = sbase + C::kVOff + st * C::kKVBytes;
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a) tma_load_3d(vdst + a * 8192, &vmap, a * 64, t * kTile, bh, v_full(st));
        issued = i + 1;
      }
      for (int i = max(0, issued - C::NSV); i < issued; ++i) wait_bounded(v_full(i % C::NSV), (i / C::NSV) & 1, p.err);
    }
  } else if (warp == kMmaS || warp == kMmaS1) {
    // ------------------------------------------------------------ S issuers: tile i into group i % 2's S
    const int sx = warp == kMmaS ? 0 : 1;  // issuer x takes the entries i % 2 == x
    if (lane == 0 && n > sx) {
      const uint32_t idS = idesc_bf16(128, 64, 0);
      bool ok = true;
      for (int i = sx; ok && i < n; i += C::kSIssuers) {
        const int st = i % C::NS, v = i & 1, j = i >> 1, b2 = j & 1;
        // NS is even, so every use of K stage st is this issuer's and it waits on the
        // stage's phases in order (see P2DualCfg).
        if (!(ok = mbar_wait(k_full(st), (i / C::NS) & 1, &abort_flag, p.err))) break;
        if (s.pages && (s.Nkv % kTile) != 0 && (int)(entry(i) & 0xFFFFu) == T - 1) {
          // paged pool: zero the K rows past Nkv of the last page before the MMA reads them
          const int nk = s.Nkv - (T - 1) * kTile, rows = kTile - nk;
          uint8_t* kst = smem + C::kKOff + st * C::kKVBytes;
          for (int x = 0; x < rows * C::kAtoms * 8; ++x) {
            const int rest = x >> 3, rr = nk + rest % rows, atom = rest / rows;
            *reinterpret_cast<uint4*>(kst + atom * 8192 + rr * 128 + (x & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        // the slot holds P of this group's entry j - 2 until its P.V has read it
        if (j >= 2 && !(ok = mbar_wait(pv_done(v, b2), ((j >> 1) - 1) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t kaddr = sbase + C::kKOff + st * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = smem_desc(sbase + C::kQOff + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(kaddr + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, kSwizzle128B);
          mma_bf16(tmem + C::kSBase + 128 * v + 64 * b2, ad, bd, idS, kk > 0);
        }
        mma_commit(s_full(v, b2));
        mma_commit(k_empty(st));  // this stage's K has been read
      }
      mma_commit(drain_s(sx));
      wait_bounded(drain_s(sx), 0, p.err);
    }
  } else if (warp == kMmaPV) {
    // ------------------------------------------------------------ PV issuer: tile i into group i % 2's O
    if (lane == 0 && n > 0) {
      const uint32_t idO = idesc_f16(128, D, 1);
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % C::NSV, v = i & 1, j = i >> 1, b2 = j & 1;
        if (!(ok = mbar_wait(p_full(v, b2), (j >> 1) & 1, &abort_flag, p.err))) break;
        if (!(ok = mbar_wait(v_full(st), (i / C::NSV) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t vaddr = sbase + C::kVOff + st * C::kKVBytes;
        // P (FP16) sits in the first 32 columns of its group's S slot: 16 keys per MMA
        const uint32_t pcol = tmem + C::kSBase + 128u * v + 64u * b2;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = smem_desc(vaddr + kk * 2048, 8192, 1024, kSwizzle128B);
          mma_f16_ts(tmem + (uint32_t)(D * v), pcol + 8u * kk, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(pv_done(v, b2));
        mma_commit(v_empty(st));  // this stage's V has been read
      }
      mma_commit(drain_pv);
      wait_bounded(drain_pv, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax: group u, one thread per row
    const int nu = (n - u + 1) / 2;  // this group's tiles: entries u, u+2, ...
    const uint32_t tO = (uint32_t)(D * u), tS = C::kSBase + 128u * u;
    const float c2 = kLog2e * rsqrtf((float)D);
    const float shift = qmu * c2;
    const int vis_last = s.causal ? pos + off : s.Nkv - 1;  // last visible key of this row
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    float m2 = -INFINITY, l2 = 0.f;
    bool ok = true;
    uint32_t e_next = nu > 0 ? entry(u) : 0u;
    for (int j = 0; j < nu; ++j) {
      const uint32_t gm = e_next >> 16;
      const int t = (int)(e_next & 0xFFFFu);
      if (j + 1 < nu) e_next = entry(2 * (j + 1) + u);
      if (!(ok = warp_wait(s_full(u, j & 1), (j >> 1) & 1))) break;
      const bool row_hot = row_valid && ((gm >> (r >> 4)) & 1u);
      const int j0 = t * kTile;
      const int nvis = row_hot ? min(kTile, vis_last + 1 - j0) : 0;  // keys j0 .. j0+nvis-1 visible
      // P (FP16, two keys per column) goes over the first 32 columns of the S slot it
      // came from; the slot's previous P had been read before S was written into it
      const uint32_t pslot = tmem + lane_base + tS + 64u * (j & 1);
      tc_fence_after();
      if (!__any_sync(0xffffffffu, nvis > 0)) {
        // neither of this warp's two groups of rows takes part in this tile: its P rows are zero
        uint32_t z[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) z[x] = 0u;
        tmem_st_x16(pslot, z);
        tmem_st_x16(pslot + 16, z);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(u, j & 1));
        continue;
      }
      uint32_t raw[64];
      tmem_ld_x32(pslot, raw);
      tmem_ld_x32(pslot + 32, raw + 32);
      tmem_wait_ld();
      float sv[64];
#pragma unroll
      for (int x = 0; x < 64; ++x) sv[x] = __uint_as_float(raw[x]);
      if (__any_sync(0xffffffffu, nvis > 0 && nvis < 64)) {
#pragma unroll
        for (int x = 0; x < 64; ++x)
          if (x >= nvis) sv[x] = -INFINITY;
      }
      float g8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        g8[k] = max3(max3(sv[8 * k], sv[8 * k + 1], sv[8 * k + 2]), max3(sv[8 * k + 3], sv[8 * k + 4], sv[8 * k + 5]),
                     fmaxf(sv[8 * k + 6], sv[8 * k + 7]));
      const float rmax = max3(max3(g8[0], g8[1], g8[2]), max3(g8[3], g8[4], g8[5]), fmaxf(g8[6], g8[7]));
      const float c = (nvis <= 0 || rmax == -INFINITY) ? -INFINITY : fmaf(rmax, c2, -shift);
      float f = 1.f;
      bool rescale = false;
      if (c > m2 + kTau2 || (m2 == -INFINITY && c > -INFINITY)) {
        if (l2 > 0.f) {
          f = ex2_approx(m2 - c);
          rescale = true;
        }
        m2 = c;
      }
      const float nb = (nvis <= 0 || m2 == -INFINITY) ? -INFINITY : -shift - m2;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[16];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int ch = 4 * hf + c4;
          p8_f16(sv + 8 * ch, c2, nb, pk + 4 * c4, ps[ch & 1], ps[2 + (ch & 1)]);
        }
        tmem_st_x16(pslot + 16u * hf, pk);
      }
      l2 = l2 * f + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      if (__any_sync(0xffffffffu, rescale)) {
        // O(u) must not be read before PV(u, j-1) has landed
        if (!(ok = warp_wait(pv_done(u, (j - 1) & 1), ((j - 1) >> 1) & 1))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(tmem + lane_base + tO + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          tmem_st_x16(tmem + lane_base + tO + c0, o);
          tmem_st_x16(tmem + lane_base + tO + c0 + 16, o + 16);
        }
      }
      tmem_wait_st();  // P (and a rescaled O) in TMEM before P.V is issued
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(u, j & 1));
    }
    // ---- epilogue: group 1 hands over (m, l); group 0 merges pass 1, group 0, group 1
    if (ok && nu > 0) ok = warp_wait(pv_done(u, (nu - 1) & 1), ((nu - 1) >> 1) & 1);
    tc_fence_after();
    if (u == 1) ml1[r] = make_float2(m2, l2);
    bool all_ok = dual_sync_and(ok);
    const int n1 = n / 2;  // group 1's tiles
    if (u == 0 && all_ok && n1 > 0)  // group 1's O is complete (waited here too, bounded)
      all_ok = warp_wait(pv_done(1, (n1 - 1) & 1), ((n1 - 1) >> 1) & 1);
    tc_fence_after();
    if (u == 0 && all_ok) {
      // the pass-1 state (none in the all-exact mode), then the two groups' states
      float m1 = -INFINITY, l1 = 0.f;
      const float* st = p.state_o ? p.state_o + ((size_t)bh * nblk * kBlockRows + P) * D : nullptr;
      if (row_valid && p.state_ml) {
        const float2 ml = p.state_ml[(size_t)bh * nblk * kBlockRows + P];
        m1 = ml.x;
        l1 = ml.y;
      }
      const float2 mlb = ml1[r];
      const float mA = m2, lA = l2, mB = mlb.x, lB = mlb.y;
      const float e1 = l1 > 0.f ? m1 : -INFINITY, eA = lA > 0.f ? mA : -INFINITY, eB = lB > 0.f ? mB : -INFINITY;
      const float M = fmaxf(e1, fmaxf(eA, eB));
      const float w1 = e1 == -INFINITY ? 0.f : exp2f(e1 - M), wA = eA == -INFINITY ? 0.f : exp2f(eA - M),
                  wB = eB == -INFINITY ? 0.f : exp2f(eB - M);
      const float L = (w1 * l1 + wA * lA) + wB * lB;
      const float invL = 1.f / L;
      const float vsc = v16_scale(__uint_as_float(p.vamax[bh]));  // O carries V / scale
      const float wAo = wA * vsc, wBo = wB * vsc;
      float* orow = p.out + (((size_t)b * s.Hq + hq) * s.Nq + pos) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t oa[32], ob[32];
        if (nu > 0) {
          tmem_ld_x32(tmem + lane_base + 0 + c0, oa);
        }
        if (n1 > 0) {
          tmem_ld_x32(tmem + lane_base + (uint32_t)D + c0, ob);
        }
        tmem_wait_ld();
        if (nu == 0) {
#pragma unroll
          for (int x = 0; x < 32; ++x) oa[x] = 0u;
        }
        if (n1 == 0) {
#pragma unroll
          for (int x = 0; x < 32; ++x) ob[x] = 0u;
        }
        if (row_valid) {
#pragma unroll
          for (int x = 0; x < 32; x += 4) {
            float4 res;
            float* rr = &res.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a1 = st ? st[c0 + x + e] : 0.f;
              rr[e] = ((w1 * a1 + wAo * __uint_as_float(oa[x + e])) + wBo * __uint_as_float(ob[x + e])) * invL;
            }
            *reinterpret_cast<float4*>(orow + c0 + x) = res;
          }
        }
      }
      if (row_valid && p.lse) {
        const float lg = M + log2f(L);
        p.lse[((size_t)b * s.Hq + hq) * s.Nq + pos] = 0.6931471805599453f * lg + qmu * rsqrtf((float)D);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// paged: the pool [num_pages][Hkv][64][d] as (channel, key in page, page * Hkv + h)
bool make_kv_map(CUtensorMap* map, const void* base, const Shape& s, CUtensorMapDataType dtype, bool paged) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<EncodeFn>(fn);
  }
  const cuuint64_t rows = paged ? (cuuint64_t)kTile : (cuuint64_t)s.Nkv;
  const cuuint64_t planes = paged ? (cuuint64_t)s.num_pages * s.Hkv : (cuuint64_t)s.BH();
  const cuuint64_t dims[3] = {(cuuint64_t)s.d, rows, planes};
  const cuuint64_t strides[2] = {(cuuint64_t)s.d * 2, rows * s.d * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Two softmax groups per block at d <= 128; at d = 256 their two O accumulators
// would take all 512 TMEM columns, so one group.
// Merges the parts of a split walk (pass2_kernel) in part order: one CTA per
// kCombineRows rows of a 128-row block (blockIdx.x: the block, blockIdx.y: its rows),
// one thread per column, the rows in turn.  The same merge as the kernel's
// epilogue: M = the largest part frame, each part weighted by 2^(m - M), O in the
// FP16-V copy's units scaled back, divided by the summed l.  In APA mode the
// pass-1 state is already in part 0, and the LSE gets each row's q.mu / sqrt(d).
constexpr int kCombineRows = 4;
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const P2Params p) {
  const Shape& s = p.s;
  const int nblk = s.nblk(), BH = s.BH(), G = s.G(), R = s.R();
  const int cta = blockIdx.x, bh = cta % BH, blk = nblk - 1 - cta / BH;
  const int b = bh / s.Hkv, h = bh % s.Hkv, c = threadIdx.x;
  const size_t item = (size_t)bh * nblk + blk;
  const float vsc = v16_scale(__uint_as_float(p.vamax[bh]));
  for (int r = blockIdx.y * kCombineRows; r < (int)(blockIdx.y + 1) * kCombineRows; ++r) {
    const int P = blk * kBlockRows + r;
    if (P >= R) break;
    const int pos = P / G, hq = h * G + P % G;
    const size_t row0 = item * p.nsplit * kBlockRows + r;
    float M = -INFINITY;
    for (int k = 0; k < p.nsplit; ++k) {
      const float2 ml = p.part_ml[row0 + (size_t)k * kBlockRows];
      M = fmaxf(M, ml.y > 0.f ? ml.x : -INFINITY);
    }
    float L = 0.f, acc = 0.f;
    for (int k = 0; k < p.nsplit; ++k) {
      const float2 ml = p.part_ml[row0 + (size_t)k * kBlockRows];
      const float w = (ml.y > 0.f && M > -INFINITY) ? exp2f(ml.x - M) : 0.f;
      L = __fmaf_rn(w, ml.y, L);
      acc = __fmaf_rn(w * vsc, p.part_o[(row0 + (size_t)k * kBlockRows) * D + c], acc);
    }
    p.out[(((size_t)b * s.Hq + hq) * s.Nq + pos) * D + c] = acc * (1.f / L);
    if (c == 0 && p.lse) {
      const float lg = M + log2f(L);
      p.lse[((size_t)b * s.Hq + hq) * s.Nq + pos] =
          0.6931471805599453f * lg + (p.mu ? p.part_qmu[item * kBlockRows + r] : 0.f);
    }
  }
}

template <int D>
cudaError_t launch_d(const P2Params& prm, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
  const int grid = prm.s.BH() * prm.s.nblk();
  cudaError_t e;
  if constexpr (D <= 128) {
    const int smem = P2DualCfg<D>::kSmem;
    if ((e = cudaFuncSetAttribute(pass2_dual_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
    pass2_dual_kernel<D><<<grid, P2DualCfg<D>::kThreads, smem, st>>>(prm, km, vm);
  } else {
    const int smem = P2Cfg<D>::kSmem;
    if ((e = cudaFuncSetAttribute(pass2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
    pass2_kernel<D><<<grid * max(1, prm.nsplit), kThreads, smem, st>>>(prm, km, vm);
    if (prm.nsplit > 1) {
      if ((e = cudaGetLastError())) return e;
      combine_kernel<D><<<dim3(grid, kBlockRows / kCombineRows), D, 0, st>>>(prm);
    }
  }
  return cudaGetLastError();
}

// Ranks the pass-2 work items by hot-list length, longest first (ties by index,
// so the order is deterministic): one block, each thread counts the items that
// precede its own.  Quadratic, so only for up to kMaxRanked items.
constexpr int kMaxRanked = 4096;
__global__ void __launch_bounds__(1024) rank_kernel(const uint32_t* __restrict__ count, int n, uint32_t* order) {
  __shared__ uint32_t c[kMaxRanked];
  for (int i = threadIdx.x; i < n; i += blockDim.x) c[i] = count[i];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t ci = c[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += (c[j] > ci) || (c[j] == ci && j < i);
    order[rank] = (uint32_t)i;
  }
}

}  // namespace

cudaError_t launch_pass2_order(const Shape& s, const Workspace& ws, cudaStream_t st) {
  const size_t n = (size_t)s.BH() * s.nblk();
  if (n > (size_t)kMaxRanked) return cudaSuccess;  // pass 2 keeps the position order
  rank_kernel<<<1, 1024, 0, st>>>(ws.hot_count, (int)n, ws.p2_order);
  return cudaGetLastError();
}

cudaError_t launch_pass2(const Shape& s, const void* q, const void* k, const void* v, const Workspace* ws, float* out,
                         float* lse, cudaStream_t st) {
  // P.V runs against the FP16 copy of V (contiguous, also for a paged K/V pool)
  (void)v;
  if (!ws || !ws->v16 || !ws->vamax) return cudaErrorInvalidValue;
  CUtensorMap km, vm;
  if (!make_kv_map(&km, k, s, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, s.pages != nullptr) ||
      !make_kv_map(&vm, ws->v16, s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, false))
    return cudaErrorInvalidValue;
  P2Params prm{};
  prm.s = s;
  prm.q = (const uint16_t*)q;
  prm.mu = ws->mu;
  prm.state_o = ws->state_o;
  prm.state_ml = ws->state_ml;
  prm.hot_list = ws->hot_list;
  prm.hot_count = ws->hot_count;
  prm.order = (size_t)s.BH() * s.nblk() <= kMaxRanked ? ws->p2_order : nullptr;
  prm.vamax = ws->vamax;
  prm.out = out;
  prm.lse = lse;
  prm.err = device_error_word();
  prm.nsplit = ws->part_o ? (ws->hot_list ? apa_split(s) : exact_split(s)) : 1;
  prm.part_o = ws->part_o;
  prm.part_ml = ws->part_ml;
  prm.part_qmu = ws->part_qmu;
  switch (s.d) {
    case 64: return launch_d<64>(prm, km, vm, st);
    case 128: return launch_d<128>(prm, km, vm, st);
    case 256: return launch_d<256>(prm, km, vm, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace apa
