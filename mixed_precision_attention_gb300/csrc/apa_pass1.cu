// apa_pass1.cu -- pass 1: every key tile in block-scaled NVFP4, with the hot test.
//
// "APA: sloppy attention, exact where it counts" (rfriedmann.de blog),
// "Pass 1: FP4 everywhere, with a hot test", per tile and 16-row group:
//   1. S = Q K^T on the FP4 tensor cores, causal mask applied;
//   2. P directly in FP4: each 16-key group gets its own scale, folded into
//      the exponent bias, so ex2 produces the quantized P;
//   3. row sums l_t of the same quantized P: by default each row's thread sums
//      its own E2M1 codes exactly in registers (a byte-permute table and dp4a);
//      with APA_FLAG_ROWSUM_MMA by one extra MMA against an E2M1 ones tile, the
//      blog's form.  Both give the exact sum of the quantized P;
//   4. the hot test: if any of the group's 16 rows has l_t > eps * lambda, the
//      tile is hot: set the mask bit, skip the PV product for the group (with the
//      value-weighted option the test is w_t * l_t > eps * lambda, w_t the tile's
//      largest key value norm over the head's mean one, after "Honest limits");
//   5. cold tiles accumulate o += P V in FP4, the cold row sum grows by l_t.
// Tile order: tile 0 (the sink), then from the causal diagonal backwards
// ("Tile order").  Frames: lazy maximum with tau = 4 ("Lazy maximum"); a hot
// tile lifts the frame only to max(m, c - 32) ("The bug: a sink that drowned
// the tail", the decoupled cold frame); the P group scale is UE4M3 ("Second
// hunt") clamped at 2^-6 ("The bug").  lambda is the running FP4 sum over every
// tile judged so far, hot ones included ("Cold verdicts are safe").
//
// Two kernels, one thread per row (TMEM lane = row) in both:
//   pass1_multi_kernel<D, U>  (the default at d <= 128): U = 3 blocks of 128
//              GQA-packed rows of one KV head per CTA, one CTA per SM.  TMEM holds
//              the three O accumulators and one S buffer the units take in turn.
//              Warps: 4 per unit (softmax), a bulk-copy producer, an S issuer and
//              a PV issuer that also writes the hot lists (see its own comment).
//   pass1_kernel<D, kOnesMma>  one block per CTA: d = 256, the residual-Q option,
//              the ones-MMA row sums, and the "wide" form of the host entry point.
//              Warps 0-3 softmax; warp 4 the bulk-copy producer (the Q blob, then
//              one 72*d-byte NVFP4 blob per tile into a 4-stage ring); warp 5 the
//              TMEM owner and MMA issuer (S, ones, PV, the scale copies, hot list).
//              With the ones-MMA row sums the softmax warps encode tile t+1 while
//              the row sums of tile t are in flight, and judge tile t afterwards
//              (tile t+1's P depends on tile t's verdict only through the frame,
//              and only when tile t lifts it); a warp whose rows lifted the frame
//              at tile t judges it first.  The issuer runs S(t+2), PV(t), ones(t+1).
//
// K/V quantization inside the launch ("What else is in the box": the next
// segment is quantized inside the launch).  When the pass-1 CTAs leave at least
// 8 SMs free, either kernel below is launched cooperatively with one CTA on
// every SM; the CTAs past the pass-1 ones run the K/V quantizer (quant_role in
// quant_tile.cuh), which publishes a flag per tile in pass 1's visiting order,
// and the producer waits (bounded) for a tile's flag before loading its blob.

#include "apa_internal.h"
#include "quant_tile.cuh"
#include "tc.cuh"

namespace apa {

namespace {

struct P1Params {
  Shape s;
  const uint8_t* kv_blob;
  const uint8_t* q_blob;
  const uint8_t* q2_blob;  // the FP4 residual term of Q, or null (one-block kernel only)
  const float* s_k;
  const float* s_v;
  const float* s_q;
  float eps;
  float* state_o;
  float2* state_ml;
  uint32_t* hot_list;
  uint32_t* hot_count;
  uint32_t* hot_mask;  // may be null
  const float* wv;     // [BH][T] value-norm weight of each tile in the hot test, or null (weight 1)
  int* err;
  // K/V quantized inside this launch (three-block kernel): CTAs n_p1.. run the
  // quantizer role; kv_ready null otherwise
  uint32_t* kv_ready;  // [BH*T] tile flags, then the quantizer's ticket counter
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  Workspace ws;
  int n_p1;
  int lse_scales;
  // test builds only (APA_TEST_HOOKS): a word nothing ever sets; when non-null the
  // producer waits on it instead of the quantizer's tile flags
  const uint32_t* test_never;
};

constexpr int kSoftWarps = 4;
constexpr int kThreads = (kSoftWarps + 2) * 32;
constexpr int kProducerWarp = kSoftWarps, kMmaWarp = kSoftWarps + 1;
// Threads of the one-block kernel.  At d = 256 twice as many: in the CTAs that run
// the K/V quantizer inside the launch, its two groups then have 192 threads each
// instead of 96, enough for it to keep ahead of pass 1 (a d = 256 tile is 64 KB of
// bf16); in the pass-1 CTAs the warps past the MMA warp stay idle.
template <int D>
constexpr int p1_threads() {
  return D >= 256 ? 2 * kThreads : kThreads;
}

template <int D>
struct P1Cfg {
  static constexpr int NS = 4;
  static constexpr int kBlob = blob_bytes(D);
  static constexpr int kQBlob = qblob_bytes(D);
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = (kQBlob + 1023) / 1024 * 1024;
  static constexpr int NP = 3;                          // P buffers (codes, scales in smem and TMEM)
  static constexpr int kPOff = kStageOff + NS * kBlob;  // NP x (128 rows x 32 B)
  static constexpr int kOnesOff = kPOff + NP * 4096;    // 16 rows x 32 B of E2M1 1.0
  static constexpr int kOnesSfOff = kOnesOff + 512;     // 512-B scale atom of UE4M3 1.0
  static constexpr int kPsfOff = kOnesSfOff + 512;      // NP x 512-B scale atoms of P
  static constexpr int kQ2Off = (kPsfOff + NP * 512 + 1023) / 1024 * 1024;  // residual Q blob
  static constexpr int kSmem = kQ2Off + kQBlob + 128;
  static constexpr uint32_t kTmemCols = D <= 128 ? 256 : 512;
  // the K/V quantizer role in this kernel: two groups of 96 threads, each with
  // double-buffered loads, or single-buffered at d = 256 (shared memory)
  static constexpr int kQuantGroups = 2, kQuantBufs = D >= 256 ? 1 : 2;
  static constexpr uint32_t kSfc = 4 * sf_chunks(D);  // TMEM columns of one K or V scale set
  // kL: the ones-MMA row sums, or (register row sums) the scales of the residual Q term
  static constexpr uint32_t kO = 0, kS = D, kL = D + 64, kSFQ = D + 80, kSFQ2 = kL;
  static_assert(4 * (D / 64) <= 16, "residual Q scales fit the row-sum columns");
  static constexpr uint32_t kSFK = kSFQ + 4 * (D / 64);  // 3 buffers (tile % 3)
  static constexpr uint32_t kSFV = kSFK + 3 * kSfc;      // 3 buffers (tile % 3)
  static constexpr uint32_t kSFP = kSFV + 3 * kSfc;      // NP buffers (tile % NP)
  static constexpr uint32_t kSFO = kSFP + 4 * NP;
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

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Eight FP32 values -> one word of eight E2M1 codes, x[0] in the lowest nibble.
__device__ __forceinline__ uint32_t pack8_e2m1(const float* x) {
  uint32_t w;
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(w)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return w;
}
// Eight P values 2^(raw * cs + nb) -> one word of eight E2M1 codes (x[0] in the
// lowest nibble); the affine step runs as four packed FP32 FMAs.
__device__ __forceinline__ uint32_t encode8(const float* x, float cs, float nb) {
  uint32_t w;
  asm("{\n.reg .b64 a0, a1, a2, a3, c2, n2;\n"
      ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "mov.b64 c2, {%9, %9};\n"
      "mov.b64 n2, {%10, %10};\n"
      "mov.b64 a0, {%1, %2};\n"
      "mov.b64 a1, {%3, %4};\n"
      "mov.b64 a2, {%5, %6};\n"
      "mov.b64 a3, {%7, %8};\n"
      "fma.rn.f32x2 a0, a0, c2, n2;\n"
      "fma.rn.f32x2 a1, a1, c2, n2;\n"
      "fma.rn.f32x2 a2, a2, c2, n2;\n"
      "fma.rn.f32x2 a3, a3, c2, n2;\n"
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
      "cvt.rn.satfinite.e2m1x2.f32 b0, y1, y0;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, y3, y2;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, y5, y4;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, y7, y6;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(w)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]), "f"(cs), "f"(nb));
  return w;
}

// Twice the E2M1 values of eight non-negative codes, summed (exact integer):
// a byte table lookup (prmt: code -> 2 * value) and two 4-byte dot products.
__device__ __forceinline__ uint32_t code_sum2(uint32_t w) {
  uint32_t lo, hi, acc;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(0x03020100u), "r"(0x0C080604u), "r"(w));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(0x03020100u), "r"(0x0C080604u), "r"(w >> 16));
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(acc) : "r"(lo), "r"(0x01010101u), "r"(0u));
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(acc) : "r"(hi), "r"(0x01010101u), "r"(acc));
  return acc;
}

// With the K/V quantizer in the same launch (lane 0 of a producer warp): waits
// until the blob of visiting position i is written; returns one past the last of
// positions i..i+7 known written (their flags read together), or -1 if the wait
// gave up (then *abort_flag is set and the timeout recorded in *err).
template <typename TileOf>
__device__ __forceinline__ int await_blobs(const uint32_t* rd, int i, int n, TileOf tile_of, int* abort_flag,
                                           int* err) {
  const unsigned long long t0 = clock64();
  while (true) {
    uint32_t got = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (i + j < n && ld_relaxed_gpu(rd + tile_of(i + j)) != 0u) got |= 1u << j;
    const int k = __ffs(~got) - 1;  // leading positions written
    if (k > 0) {
      __threadfence();             // acquire: the blob stores come before the flags
      fence_proxy_async_global();  // and before the bulk copies that read them
      return i + k;
    }
    if (*(volatile int*)abort_flag) return -1;
    if (clock64() - t0 > APA_WAIT_LIMIT_CYCLES) {
      *(volatile int*)abort_flag = 1;
      if (err) atomicCAS(err, 0, APA_DEVERR_TIMEOUT);
      return -1;
    }
    __nanosleep(128);
  }
}

// The producer's wait for tiles i.. of head bh: on the quantizer's flags, or (test
// builds) on a word nothing sets, so that the wait runs out.
template <typename TileOf>
__device__ __forceinline__ int await_tiles(const P1Params& p, int bh, int T, int i, int n, TileOf tile_of,
                                           int* abort_flag) {
  if (p.test_never) return await_blobs(p.test_never, i, n, [](int) { return 0; }, abort_flag, p.err);
  return await_blobs(p.kv_ready + (size_t)bh * T, i, n, tile_of, abort_flag, p.err);
}

// What a row keeps between encoding a tile and judging it.
struct Pending {
  float c, mt;
  uint32_t sfw;
  bool empty, lift;
};

// kOnesMma: the tile row sums come from an extra MMA of P against an E2M1 ones
// tile (the blog's form: the softmax warps encode tile t+1 while the row sums
// of tile t are in flight).  Otherwise each thread sums its own row's quantized
// P exactly in registers (a byte table lookup of the codes), so the hot test
// follows the encode directly, a hot group's P scales are written as zero, and
// a tile costs the softmax warps one wait and two arrives.
template <int D, bool kOnesMma>
__global__ void __launch_bounds__(p1_threads<D>(), (D <= 128 ? 2 : 1)) pass1_kernel(const P1Params p) {
  using C = P1Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  if (!kOnesMma && p.kv_ready && (int)blockIdx.x >= p.n_p1) {
    // the K/V quantizer, in groups that each keep a tile in flight: the tiles in
    // the order the pass-1 CTAs below visit them
    constexpr int kGroup = p1_threads<D>() / C::kQuantGroups;
    static_assert(kGroup % 32 == 0 && kGroup % (D / 16) == 0 && p1_threads<D>() % C::kQuantGroups == 0,
                  "quantizer groups of whole warps");
    const int g = threadIdx.x / kGroup;
    quant_role(p.s, p.k_raw, p.v_raw, p.ws, p.kv_ready, p.kv_ready + (size_t)p.s.BH() * p.s.T(), p.lse_scales != 0,
               smem + g * quant_role_smem(D, C::kQuantBufs), p.err, g, threadIdx.x % kGroup, kGroup, C::kQuantBufs);
    return;
  }
  // barriers: q_full, blob_full[4], blob_empty[4], s_full, s_free, p_full[2], l_full, dec[2], pv_done[2], drain
  __shared__ __align__(8) uint64_t bars[19];
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
  const uint32_t drain = bar0 + 8u * 18;
  auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;  // already complete: no spin
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
    for (int i = 0; i < 19; ++i) {
      const bool per_warp = (i == 10) || (i >= 11 && i <= 12) || (i >= 14 && i <= 15);  // s_free, p_full, dec
      mbar_init(bar0 + 8u * i, per_warp ? (uint32_t)kSoftWarps : 1u);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x < 128) {
    // the ones tile (E2M1 1.0 = code 2) and its scale atom (UE4M3 1.0 = 0x38)
    reinterpret_cast<uint2*>(smem + C::kOnesOff)[threadIdx.x] =
        threadIdx.x < 64 ? make_uint2(0x22222222u, 0x22222222u) : make_uint2(0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ bulk-copy producer
    if (lane == 0) {
      const uint8_t* qsrc = p.q_blob + ((size_t)bh * nblk + blk) * C::kQBlob;
      const bool q2 = !kOnesMma && p.q2_blob;
      mbar_arrive_expect_tx(q_full, q2 ? 2 * C::kQBlob : C::kQBlob);
      bulk_g2s(sbase + C::kQOff, qsrc, C::kQBlob, q_full);
      if (q2) bulk_g2s(sbase + C::kQ2Off, p.q2_blob + ((size_t)bh * nblk + blk) * C::kQBlob, C::kQBlob, q_full);
      int issued = 0, written = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(blob_empty(st), ((i / C::NS) - 1) & 1, &abort_flag, p.err)) break;
        if (!kOnesMma && p.kv_ready && i >= written &&
            (written = await_tiles(p, bh, T, i, n, tile_of, &abort_flag)) < 0)
          break;
        const uint8_t* src = p.kv_blob + ((size_t)bh * T + tile_of(i)) * C::kBlob;
        mbar_arrive_expect_tx(blob_full(st), C::kBlob);
        bulk_g2s(sbase + C::kStageOff + st * C::kBlob, src, C::kBlob, blob_full(st));
        issued = i + 1;
      }
      // Every copy issued lands before the CTA exits, also when another warp gave up
      // after this loop ended.  Normally all have landed (and no copy reused their
      // stage since), so these parity waits return at once.
      wait_bounded(q_full, 0, p.err);
      for (int i = max(0, issued - C::NS); i < issued; ++i) wait_bounded(blob_full(i % C::NS), (i / C::NS) & 1, p.err);
    }
  } else if (warp == kMmaWarp) {
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
        if (!kOnesMma && p.q2_blob)
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tmem_cp_32x128b_x4(tmem + C::kSFQ2 + 4 * a,
                               smem_desc(sbase + C::kQ2Off + qblob_sf(D) + 512 * a, 128, 128, 0));
        tmem_cp_32x128b_x4(tmem + C::kSFO, smem_desc(sbase + C::kOnesSfOff, 128, 128, 0));
      }
      // S(i) into the single S buffer once tile i-1 has been read out of it
      auto issue_s = [&](int i) -> bool {
        const int st = i % C::NS;
        if (!mbar_wait(blob_full(st), (i / C::NS) & 1, &abort_flag, p.err)) return false;
        if (i >= 1 && !mbar_wait(s_free, (i - 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t blob = sbase + C::kStageOff + st * C::kBlob;
        const uint32_t sfk = tmem + C::kSFK + C::kSfc * (i % 3);
        const uint32_t sfv = tmem + C::kSFV + C::kSfc * (i % 3);
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
        if (!kOnesMma && p.q2_blob) {
          // the residual term of Q, accumulated into the same S against the same K
#pragma unroll
          for (int kk = 0; kk < D / 64; ++kk) {
            const uint64_t ad = smem_desc(sbase + C::kQ2Off + 256 * kk, 128, 4 * D, 0);
            const uint64_t bd = smem_desc(blob + blob_kcodes(D) + 256 * kk, 128, 4 * D, 0);
            mma_nvf4(tmem + C::kS, ad, bd, idS, tmem + C::kSFQ2 + 4 * kk, sfk + 4 * (kk >> 1) + 2 * (kk & 1), 1);
          }
        }
        mma_commit(s_full);
        return true;
      };
      // ones(i): the FP4 row sums of P(i)
      auto issue_ones = [&](int i) -> bool {
        if (!mbar_wait(p_full(i & 1), (i >> 1) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const int pb = i % C::NP;
        tmem_cp_32x128b_x4(tmem + C::kSFP + 4 * pb, smem_desc(sbase + C::kPsfOff + 512 * pb, 128, 128, 0));
        mma_nvf4(tmem + C::kL, smem_desc(sbase + C::kPOff + 4096 * pb, 128, 256, 0),
                 smem_desc(sbase + C::kOnesOff, 128, 256, 0), idL, tmem + C::kSFP + 4 * pb, tmem + C::kSFO, 0);
        mma_commit(l_full);
        return true;
      };
      uint32_t pv_issued = 0;
      if (!kOnesMma) {
        // S(i+1) as soon as S(i) has been read out; PV(i) once P(i) and its verdicts are in
        if (ok) ok = issue_s(0);
        for (int i = 0; ok && i < n; ++i) {
          if (i + 1 < n && !(ok = issue_s(i + 1))) break;
          if (!(ok = mbar_wait(p_full(i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
          tc_fence_after();
          const uint32_t hot = gbits[i & 1][0] | gbits[i & 1][1] | gbits[i & 1][2] | gbits[i & 1][3];
          if (hot) list[count++] = (uint32_t)tile_of(i) | (hot << 16);
          if ((hot | invalid_groups) != 0xFFu) {
            const uint32_t blob = sbase + C::kStageOff + (i % C::NS) * C::kBlob;
            const int pb = i % C::NP;
            tmem_cp_32x128b_x4(tmem + C::kSFP + 4 * pb, smem_desc(sbase + C::kPsfOff + 512 * pb, 128, 128, 0));
            mma_nvf4(tmem + C::kO, smem_desc(sbase + C::kPOff + 4096 * pb, 128, 256, 0),
                     smem_desc(blob + blob_vcodes(D), 128, 256, 0), idO, tmem + C::kSFP + 4 * pb,
                     tmem + C::kSFV + C::kSfc * (i % 3), pv_issued > 0);
            ++pv_issued;
          }
          mma_commit(pv_done(i & 1));
          mma_commit(blob_empty(i % C::NS));
        }
        ok = false;  // skip the ones-MMA schedule below
      }
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      if (ok) ok = issue_ones(0);
      for (int i = 0; ok && i < n; ++i) {
        if (i + 2 < n && !(ok = issue_s(i + 2))) break;
        if (!(ok = mbar_wait(dec(i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t hot = gbits[i & 1][0] | gbits[i & 1][1] | gbits[i & 1][2] | gbits[i & 1][3];
        if (hot) list[count++] = (uint32_t)tile_of(i) | (hot << 16);
        if ((hot | invalid_groups) != 0xFFu) {
          const uint32_t blob = sbase + C::kStageOff + (i % C::NS) * C::kBlob;
          const int pb = i % C::NP;
          if (hot)  // the hot groups' P scales were zeroed in smem: copy them again for PV
            tmem_cp_32x128b_x4(tmem + C::kSFP + 4 * pb, smem_desc(sbase + C::kPsfOff + 512 * pb, 128, 128, 0));
          mma_nvf4(tmem + C::kO, smem_desc(sbase + C::kPOff + 4096 * pb, 128, 256, 0),
                   smem_desc(blob + blob_vcodes(D), 128, 256, 0), idO, tmem + C::kSFP + 4 * pb,
                   tmem + C::kSFV + C::kSfc * (i % 3), pv_issued > 0);
          ++pv_issued;
        }
        mma_commit(pv_done(i & 1));
        mma_commit(blob_empty(i % C::NS));
        if (i + 1 < n && !(ok = issue_ones(i + 1))) break;
      }
      p.hot_count[(size_t)bh * nblk + blk] = count;
      mma_commit(drain);
      wait_bounded(drain, 0, p.err);
    }
  } else if (warp < kSoftWarps) {
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
    const int ngroups = s.ngroups(), nwords = (T + 31) / 32;
    float m = -INFINITY, lam = 0.f, l = 0.f;
    bool ok = true;

    // Encodes P of tile i in the frame that follows from the current m and
    // hands it to the MMA issuer (codes in smem, scales in TMEM).
    auto encode = [&](int i, Pending& pd) -> bool {
      const int t = tile_of(i), j0 = t * kTile;
      const int nvis = valid ? min(kTile, vis_last + 1 - j0) : 0;
      if (!warp_wait(s_full, i & 1)) return false;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld_x32(tmem + lane_base + C::kS, sr);
      tmem_ld_x32(tmem + lane_base + C::kS + 32, sr + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      float raw[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) raw[j] = __uint_as_float(sr[j]);
      if (__any_sync(0xffffffffu, nvis < kTile)) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j >= nvis) raw[j] = -INFINITY;
      }
      float g[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = max3(raw[16 * k], raw[16 * k + 1], raw[16 * k + 2]);
#pragma unroll
        for (int j = 3; j < 15; j += 2) a = max3(a, raw[16 * k + j], raw[16 * k + j + 1]);
        g[k] = fmaxf(a, raw[16 * k + 15]);
      }
      pd.c = fmaxf(fmaxf(g[0], g[1]), fmaxf(g[2], g[3])) * cs;  // tile max, log2 units
      pd.empty = (pd.c == -INFINITY);
      pd.mt = (pd.c > m + kTau) ? pd.c : m;  // candidate frame (lazy maximum)
      pd.lift = !pd.empty && pd.mt != m;
      uint32_t pw[8];
      pd.sfw = 0x08080808u;  // 2^-6 where nothing is visible
      if (!pd.empty) {
        pd.sfw = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t sc = cvt_ue4m3(ex2_approx(fmaf(g[k], cs, -pd.mt)) * (1.f / 6.f));
          sc = max(sc, 8u);  // clamp the group scale at 2^-6
          pd.sfw |= sc << (8 * k);
          const float nb = -(pd.mt + lg2_approx(ue4m3_value(sc)));
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = ex2_approx(fmaf(raw[16 * k + 8 * w + e], cs, nb));
            pw[2 * k + w] = pack8_e2m1(y);
          }
        }
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) pw[w] = 0u;
      }
      // P buffer i % 3 was last read by PV(i-3) and the ones-MMA of tile i-3; both
      // completed before the ones-MMA of tile i-1, which judge(i-1) waited for
      // (tcgen05 ops of the issuing thread complete in order and a commit covers
      // all earlier ones), so the buffer is free without another wait.
      const int pbuf = i % C::NP;
      uint8_t* pb = smem + C::kPOff + 4096 * pbuf + (r >> 3) * 256 + (r & 7) * 16;
      *reinterpret_cast<uint4*>(pb) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(pb + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      *reinterpret_cast<uint32_t*>(smem + C::kPsfOff + 512 * pbuf + sf_atom_off(r, 0)) = pd.sfw;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(i & 1));
      return true;
    };

    // Judges tile i from its FP4 row sums and commits frame, lambda and l.
    // `lifted`: some row of this warp moved its frame at tile i (else every row
    // keeps m, so lambda += l_t and, if cold, l += l_t: no exponentials, no rescale).
    auto judge = [&](int i, const Pending& pd, bool lifted) -> bool {
      const int t = tile_of(i);
      const float wt = p.wv ? __ldg(p.wv + (size_t)bh * T + t) : 1.f;
      if (!warp_wait(l_full, i & 1)) return false;
      tc_fence_after();
      uint32_t lb;
      tmem_ld_x1(tmem + lane_base + C::kL, lb);
      tmem_wait_ld();
      const float ell = __uint_as_float(lb);
      // hot test: w_t * l_t (in the committed frame) > eps * lambda; thr is -1 at eps = 0
      // (every visible tile hot) and NaN at eps = inf with lambda = 0 (never hot)
      const float thr = eps == 0.f ? -1.f : eps * lam;
      const float ellw = ell * wt;
      bool vote;
      if (!lifted) vote = valid && !pd.empty && ellw > thr;
      else vote = valid && !pd.empty && !eps_inf &&
                  ((m == -INFINITY) ? (eps == 0.f || ellw > 0.f) : (ellw * ex2_approx(pd.mt - m) > thr));
      const uint32_t bal = __ballot_sync(0xffffffffu, vote);
      const bool hot_lo = (bal & 0x0000FFFFu) != 0, hot_hi = (bal & 0xFFFF0000u) != 0;
      const bool hot = lane < 16 ? hot_lo : hot_hi;
      if (!lifted) {
        if (!pd.empty) {
          lam += ell;
          if (!hot) l += ell;
        }
      } else {
        bool rescale = false;
        float f = 1.f;
        if (!pd.empty) {
          const float l_before = l;
          float mn;
          if (hot) {
            mn = fmaxf(m, pd.c - kColdOffset);
            f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
            lam = lam * f + ell * ex2_approx(pd.mt - mn);
            l *= f;
          } else {
            mn = pd.mt;
            f = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
            lam = lam * f + ell;
            l = l * f + ell;
          }
          rescale = (f != 1.f) && (l_before > 0.f);
          m = mn;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          // PV(i-1) has landed: it was issued before the ones-MMA of tile i, waited for above
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
          tmem_wait_st();
        }
      }
      if (hot) {  // a hot group's P drops out of PV: zero its scales in smem
        *reinterpret_cast<uint32_t*>(smem + C::kPsfOff + 512 * (i % C::NP) + sf_atom_off(r, 0)) = 0u;
        fence_proxy_async_smem();
      }
      if (lane == 0) gbits[i & 1][warp] = ((uint32_t)hot_lo << (2 * warp)) | ((uint32_t)hot_hi << (2 * warp + 1));
      if (p.hot_mask && (lane == 0 || lane == 16) && hot) {
        const int grp = (p0 + 32 * warp + lane) / kGroupRows;
        if (grp < ngroups) atomicOr(&p.hot_mask[((size_t)bh * ngroups + grp) * nwords + t / 32], 1u << (t % 32));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dec(i & 1));
      return true;
    };

    if (kOnesMma) {
      Pending cur, nxt;
      ok = encode(0, cur);
      for (int i = 0; ok && i < n; ++i) {
        const bool lifted = __any_sync(0xffffffffu, cur.lift);
        if (i + 1 < n) {
          // tile i+1 can be encoded before tile i is judged unless a row of this
          // warp lifted its frame at tile i (then m after tile i depends on the verdict)
          if (!lifted) {
            if (!(ok = encode(i + 1, nxt))) break;
            if (!(ok = judge(i, cur, false))) break;
          } else {
            if (!(ok = judge(i, cur, true))) break;
            if (!(ok = encode(i + 1, nxt))) break;
          }
          cur = nxt;
        } else {
          ok = judge(i, cur, lifted);
        }
      }
    } else {
      // ---- row sums in registers: encode, sum, judge and hand over, one tile at a time
      for (int i = 0; ok && i < n; ++i) {
        const int t = tile_of(i), j0 = t * kTile;
        const int nvis = valid ? min(kTile, vis_last + 1 - j0) : 0;
        const float wt = p.wv ? __ldg(p.wv + (size_t)bh * T + t) : 1.f;
        if (!(ok = warp_wait(s_full, i & 1))) break;
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld_x32(tmem + lane_base + C::kS, sr);
        tmem_ld_x32(tmem + lane_base + C::kS + 32, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        float raw[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) raw[j] = __uint_as_float(sr[j]);
        if (__any_sync(0xffffffffu, nvis < kTile)) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (j >= nvis) raw[j] = -INFINITY;
        }
        float g[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a = max3(raw[16 * k], raw[16 * k + 1], raw[16 * k + 2]);
#pragma unroll
          for (int j = 3; j < 15; j += 2) a = max3(a, raw[16 * k + j], raw[16 * k + j + 1]);
          g[k] = fmaxf(a, raw[16 * k + 15]);
        }
        const float c = fmaxf(fmaxf(g[0], g[1]), fmaxf(g[2], g[3])) * cs;  // tile max, log2 units
        const bool empty = (c == -INFINITY);
        const float mt = (c > m + kTau) ? c : m;  // candidate frame (lazy maximum)
        uint32_t pw[8];
        uint32_t sfw = 0x08080808u;  // 2^-6 where nothing is visible
        float ell = 0.f;             // l_t: exact sum of the quantized P of this row
        if (!empty) {
          // the four group scales, clamped at 2^-6 (code 8), converted and decoded in pairs
          float gs[4], scv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) gs[k] = ex2_approx(fmaf(g[k], cs, -mt)) * (1.f / 6.f);
          sfw = cvt_ue4m3x4_min(gs[0], gs[1], gs[2], gs[3], 8u);
          ue4m3x4_values(sfw, scv);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float nb = -(mt + lg2_approx(scv[k]));
#pragma unroll
            for (int w = 0; w < 2; ++w) pw[2 * k + w] = encode8(raw + 16 * k + 8 * w, cs, nb);
            ell = fmaf((float)(code_sum2(pw[2 * k]) + code_sum2(pw[2 * k + 1])), 0.5f * scv[k], ell);
          }
        } else {
#pragma unroll
          for (int w = 0; w < 8; ++w) pw[w] = 0u;
        }
        // hot test: w_t * l_t (in the committed frame) > eps * lambda
        const bool lift = !empty && mt != m;
        const bool lifted = __any_sync(0xffffffffu, lift);
        const float thr = eps == 0.f ? -1.f : eps * lam;
        const float ellw = ell * wt;
        bool vote;
        if (!lifted) vote = valid && !empty && ellw > thr;
        else vote = valid && !empty && !eps_inf &&
                    ((m == -INFINITY) ? (eps == 0.f || ellw > 0.f) : (ellw * ex2_approx(mt - m) > thr));
        const uint32_t bal = __ballot_sync(0xffffffffu, vote);
        const bool hot_lo = (bal & 0x0000FFFFu) != 0, hot_hi = (bal & 0xFFFF0000u) != 0;
        const bool hot = lane < 16 ? hot_lo : hot_hi;
        if (!lifted) {
          if (!empty) {
            lam += ell;
            if (!hot) l += ell;
          }
        } else {
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
          if (__any_sync(0xffffffffu, rescale)) {
            // O must not be touched before PV(i-1) has landed
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
            tmem_wait_st();
          }
        }
        // P buffer i % 3 was last read by PV(i-3), issued before S(i), whose completion
        // was waited for above: free without another wait.  A hot group's scales are
        // zero, so its rows drop out of PV.
        const int pbuf = i % C::NP;
        uint8_t* pbp = smem + C::kPOff + 4096 * pbuf + (r >> 3) * 256 + (r & 7) * 16;
        *reinterpret_cast<uint4*>(pbp) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        *reinterpret_cast<uint4*>(pbp + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
        *reinterpret_cast<uint32_t*>(smem + C::kPsfOff + 512 * pbuf + sf_atom_off(r, 0)) = hot ? 0u : sfw;
        if (lane == 0) gbits[i & 1][warp] = ((uint32_t)hot_lo << (2 * warp)) | ((uint32_t)hot_hi << (2 * warp + 1));
        if (p.hot_mask && (lane == 0 || lane == 16) && hot) {
          const int grp = (p0 + 32 * warp + lane) / kGroupRows;
          if (grp < ngroups) atomicOr(&p.hot_mask[((size_t)bh * ngroups + grp) * nwords + t / 32], 1u << (t % 32));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(i & 1));
      }
    }
    // ---- epilogue: the pass-1 state (o scaled by s_v, frame m, cold sum l)
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// Pass 1 with U row blocks of one KV head per CTA (d <= 128).
//
// TMEM holds U output accumulators (U * d columns) and one S buffer that the
// units take in turn; at d = 128 and U = 3 that is all 512 columns, so one CTA
// per SM keeps 3 blocks (384 rows) in flight instead of 2.  The units walk one
// common tile order 0, T_max, ..., 1 (T_max: the last tile any of them sees; a
// tile past a unit's own diagonal is fully masked for it, so a no-op) and share
// each K/V blob and its scales.  Per unit the softmax work is the
// register-row-sum form of the single-block kernel.
//
// Two warps issue the tensor-core work, so that neither issue stream is a
// serial bottleneck for three units: the S warp issues S(0,i), S(1,i), ... in
// the order in which the units hand the S buffer on; the PV warp issues
// PV(u,i) as each unit publishes P(u,i).
constexpr int kUnits = 3;  // 128-row blocks per CTA of the multi-block kernel
template <int D, int U>
struct P1MCfg {
  static constexpr int NS = 4;
  static constexpr int kBlob = blob_bytes(D);
  static constexpr int kQBlob = qblob_bytes(D);
  static constexpr int kQStride = (kQBlob + 1023) / 1024 * 1024;
  static constexpr int kStageOff = U * kQStride;
  static constexpr int kPOff = kStageOff + NS * kBlob;  // [U][2] x (128 rows x 32 B)
  static constexpr int kSmem = kPOff + U * 2 * 4096 + 128;  // (P's scales go straight to TMEM)
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSfc = 4 * sf_chunks(D);
  static constexpr uint32_t kS = U * D;
  static constexpr uint32_t kSFQ = kS + 64;                   // U x 4 * (D/64)
  static constexpr uint32_t kSFK = kSFQ + U * 4 * (D / 64);   // 2 buffers (tile % 2)
  static constexpr uint32_t kSFV = kSFK + 2 * kSfc;           // 2 buffers (tile % 2)
  static constexpr uint32_t kSFP = kSFV + 2 * kSfc;           // [U][2] buffers (tile % 2)
  static_assert(kSFP + 8 * U <= kTmemCols, "TMEM budget");
  static constexpr int kThreads = (4 * U + 3) * 32;
  // thread groups of the K/V quantizer role (each a multiple of d/16 threads)
  static constexpr int kQuantGroups = 3;
  static_assert(kThreads % kQuantGroups == 0 && (kThreads / kQuantGroups) % (D / 16) == 0 &&
                    (kThreads / kQuantGroups) % 32 == 0 && kQuantGroups <= kQuantRoleGroups,
                "quantizer groups");
};

template <int D, int U>
__global__ void __launch_bounds__(P1MCfg<D, U>::kThreads, 1) pass1_multi_kernel(const P1Params p) {
  using C = P1MCfg<D, U>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  if (p.kv_ready && (int)blockIdx.x >= p.n_p1) {
    // the K/V quantizer, in groups that each keep a tile in flight: the tiles in
    // the order the pass-1 CTAs below visit them
    constexpr int kGroup = C::kThreads / C::kQuantGroups;
    const int g = threadIdx.x / kGroup;
    quant_role(p.s, p.k_raw, p.v_raw, p.ws, p.kv_ready, p.kv_ready + (size_t)p.s.BH() * p.s.T(), p.lse_scales != 0,
               smem + g * quant_role_smem(D), p.err, g, threadIdx.x % kGroup, kGroup, 2);
    return;
  }
  // barriers: q_full, blob_full[NS], blob_empty[NS], s_full[U], s_free[U], p_full[U][2], pv_done[U][2],
  // drain_s, drain_pv
  constexpr int kBars = 1 + 2 * C::NS + 6 * U + 2;
  __shared__ __align__(8) uint64_t bars[kBars];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t gbits[U][2][4];

  const Shape& s = p.s;
  const int nblk = s.nblk(), BH = s.BH(), G = s.G(), R = s.R(), T = s.T(), off = s.off();
  const int ngrp = (nblk + U - 1) / U;
  const int bh = blockIdx.x % BH, grp = ngrp - 1 - (int)(blockIdx.x / BH);  // heavy (late) blocks first
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kProd = 4 * U, kMmaS = 4 * U + 1, kMmaPV = 4 * U + 2;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0;
  auto blob_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto blob_empty = [&](int st) { return bar0 + 8u * (1 + C::NS + st); };
  auto s_full = [&](int u) { return bar0 + 8u * (1 + 2 * C::NS + u); };
  auto s_free = [&](int u) { return bar0 + 8u * (1 + 2 * C::NS + U + u); };
  auto p_full = [&](int u, int par) { return bar0 + 8u * (1 + 2 * C::NS + 2 * U + 2 * u + par); };
  auto pv_done = [&](int u, int par) { return bar0 + 8u * (1 + 2 * C::NS + 4 * U + 2 * u + par); };
  const uint32_t drain_s = bar0 + 8u * (kBars - 2), drain_pv = bar0 + 8u * (kBars - 1);
  auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    const bool okl = mbar_wait(bar, parity, &abort_flag, p.err);
    return __all_sync(0xffffffffu, okl);
  };

  // the units: blocks grp*U + u of this head; the common tile order ends at T_max
  const int blk_last = min(nblk, (grp + 1) * U) - 1;
  const int last_row = min(R, (blk_last + 1) * kBlockRows) - 1;
  const int t_hi = s.causal ? min(T - 1, (last_row / G + off) / kTile) : T - 1;
  const int n = t_hi + 1;
  auto tile_of = [&](int i) { return i == 0 ? 0 : t_hi + 1 - i; };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < kBars; ++i) {
      const int j = i - (1 + 2 * C::NS);
      uint32_t count = 1;
      if (j >= U && j < 4 * U) count = 4;           // s_free, p_full: the unit's four warps
      if (i >= 1 + C::NS && i < 1 + 2 * C::NS) count = 2;  // blob_empty: both issuers
      mbar_init(bar0 + 8u * i, count);
    }
    fence_mbar_init();
  }
  if (warp == kMmaS) {
    tmem_alloc(smem_u32(&tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kProd) {
    // ------------------------------------------------------------ bulk-copy producer
    if (lane == 0) {
      uint32_t qbytes = 0;
      for (int u = 0; u < U; ++u)
        if (grp * U + u < nblk) qbytes += C::kQBlob;
      mbar_arrive_expect_tx(q_full, qbytes);
      for (int u = 0; u < U; ++u)
        if (grp * U + u < nblk)
          bulk_g2s(sbase + u * C::kQStride, p.q_blob + ((size_t)bh * nblk + grp * U + u) * C::kQBlob, C::kQBlob,
                   q_full);
      int issued = 0, written = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(blob_empty(st), ((i / C::NS) - 1) & 1, &abort_flag, p.err)) break;
        if (p.kv_ready && i >= written &&
            (written = await_tiles(p, bh, T, i, n, tile_of, &abort_flag)) < 0)
          break;
        mbar_arrive_expect_tx(blob_full(st), C::kBlob);
        bulk_g2s(sbase + C::kStageOff + st * C::kBlob, p.kv_blob + ((size_t)bh * T + tile_of(i)) * C::kBlob,
                 C::kBlob, blob_full(st));
        issued = i + 1;
      }
      // Every copy issued lands before the CTA exits, also when another warp gave up
      // after this loop ended.  Normally all have landed (and no copy reused their
      // stage since), so these parity waits return at once.
      wait_bounded(q_full, 0, p.err);
      for (int i = max(0, issued - C::NS); i < issued; ++i) wait_bounded(blob_full(i % C::NS), (i / C::NS) & 1, p.err);
    }
  } else if (warp == kMmaS) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      const uint32_t idS = idesc_nvf4(128, 64);
      bool ok = mbar_wait(q_full, 0, &abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tmem_cp_32x128b_x4(tmem + C::kSFQ + 4 * ((D / 64) * u + a),
                               smem_desc(sbase + u * C::kQStride + qblob_sf(D) + 512 * a, 128, 128, 0));
      }
      // K scales of tile i into TMEM buffer i % 2, once its blob has landed
      auto load_sfk = [&](int i) -> bool {
        const int st = i % C::NS;
        if (!mbar_wait(blob_full(st), (i / C::NS) & 1, &abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t blob = sbase + C::kStageOff + st * C::kBlob;
#pragma unroll
        for (int c = 0; c < sf_chunks(D); ++c)
          tmem_cp_32x128b_x4(tmem + C::kSFK + C::kSfc * (i & 1) + 4 * c,
                             smem_desc(blob + blob_ksf(D) + 512 * c, 128, 128, 0));
        return true;
      };
      // operand descriptors of unit 0 / stage 0; the others differ only in the start
      // address field (address >> 4, no carry out of it inside shared memory)
      const uint64_t qd0 = smem_desc(sbase, 128, 4 * D, 0);
      const uint64_t kd0 = smem_desc(sbase + C::kStageOff + blob_kcodes(D), 128, 4 * D, 0);
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % C::NS;
        const uint32_t sfk = tmem + C::kSFK + C::kSfc * (i & 1);
        for (int u = 0; ok && u < U; ++u) {
          // S(u, i) once the previous user of the S buffer has read it out
          if (u > 0) {
            if (!(ok = mbar_spin_wait(s_free(u - 1), i & 1, &abort_flag, p.err))) break;
          } else {
            // the K scales of tile i: their buffer was last read by S(*, i-2)
            if (!(ok = load_sfk(i))) break;
            if (i > 0 && !(ok = mbar_spin_wait(s_free(U - 1), (i - 1) & 1, &abort_flag, p.err))) break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 64; ++kk)
            mma_nvf4(tmem + C::kS, qd0 + ((uint32_t)(u * C::kQStride + 256 * kk) >> 4),
                     kd0 + ((uint32_t)(st * C::kBlob + 256 * kk) >> 4), idS, tmem + C::kSFQ + 4 * ((D / 64) * u + kk),
                     sfk + 4 * (kk >> 1) + 2 * (kk & 1), kk > 0);
          mma_commit(s_full(u));
        }
        if (ok) mma_commit(blob_empty(st));
      }
      mma_commit(drain_s);
      wait_bounded(drain_s, 0, p.err);
    }
  } else if (warp == kMmaPV) {
    // ------------------------------------------------------------ PV issuer and hot lists
    if (lane == 0) {
      const uint32_t idO = idesc_nvf4(128, D);
      uint32_t count[U], pv_issued[U];
      for (int u = 0; u < U; ++u) count[u] = pv_issued[u] = 0;
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % C::NS;
        const uint32_t blob = sbase + C::kStageOff + st * C::kBlob;
        const uint32_t sfv = tmem + C::kSFV + C::kSfc * (i & 1);
        for (int u = 0; ok && u < U; ++u) {
          if (!(ok = mbar_wait(p_full(u, i & 1), (i >> 1) & 1, &abort_flag, p.err))) break;
          if (u == 0) {
            // V scales of tile i; their buffer was last read by PV(*, i-2), covered by the
            // commit of pv_done(U-1, i-2)
            if (!(ok = mbar_wait(blob_full(st), (i / C::NS) & 1, &abort_flag, p.err))) break;
            if (i >= 2 && !(ok = mbar_wait(pv_done(U - 1, i & 1), ((i - 2) >> 1) & 1, &abort_flag, p.err))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < sf_chunks(D); ++c)
              tmem_cp_32x128b_x4(sfv + 4 * c, smem_desc(blob + blob_vsf(D) + 512 * c, 128, 128, 0));
          }
          tc_fence_after();
          const int blk = grp * U + u;
          if (blk < nblk) {
            const int nvg = (min(R, (blk + 1) * kBlockRows) - blk * kBlockRows + kGroupRows - 1) / kGroupRows;
            const uint32_t invalid = 0xFFu & ~((1u << nvg) - 1u);
            const uint32_t hot = gbits[u][i & 1][0] | gbits[u][i & 1][1] | gbits[u][i & 1][2] | gbits[u][i & 1][3];
            if (hot) p.hot_list[((size_t)bh * nblk + blk) * T + count[u]++] = (uint32_t)tile_of(i) | (hot << 16);
            if ((hot | invalid) != 0xFFu) {
              // P buffer (u, i % 2) and its TMEM scales were last read by PV(u, i-2); unit u
              // waited for it before writing P(u, i) and its scales
              const int pb = 2 * u + (i & 1);
              mma_nvf4(tmem + D * u, smem_desc(sbase + C::kPOff + 4096 * pb, 128, 256, 0),
                       smem_desc(blob + blob_vcodes(D), 128, 256, 0), idO, tmem + C::kSFP + 4 * pb, sfv,
                       pv_issued[u] > 0);
              ++pv_issued[u];
            }
          }
          mma_commit(pv_done(u, i & 1));
        }
        if (ok) mma_commit(blob_empty(st));
      }
      for (int u = 0; u < U; ++u)
        if (grp * U + u < nblk) p.hot_count[(size_t)bh * nblk + grp * U + u] = count[u];
      mma_commit(drain_pv);
      wait_bounded(drain_pv, 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ one thread per row of unit u
    const int u = warp >> 2, qw = warp & 3;
    const int blk = grp * U + u;
    const int r = qw * 32 + lane, P = blk * kBlockRows + r;
    const bool valid = blk < nblk && P < R;
    const int pos = valid ? P / G : 0;
    const int hq = h * G + (valid ? P % G : 0);
    const float cs = p.s_q[b * s.Hq + hq] * p.s_k[bh] * (kLog2e * rsqrtf((float)D));
    const int vis_last = s.causal ? pos + off : s.Nkv - 1;
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    const uint32_t tO = tmem + lane_base + D * u;
    const float eps = p.eps;
    const bool eps_inf = isinf(eps);
    const int ngroups = s.ngroups(), nwords = (T + 31) / 32;
    float m = -INFINITY, lam = 0.f, l = 0.f;
    bool ok = true;
    for (int i = 0; ok && i < n; ++i) {
      const int t = tile_of(i), j0 = t * kTile;
      const int nvis = valid ? min(kTile, vis_last + 1 - j0) : 0;
      const float wt = p.wv ? __ldg(p.wv + (size_t)bh * T + t) : 1.f;
      if (!(ok = warp_wait(s_full(u), i & 1))) break;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld_x32(tmem + lane_base + C::kS, sr);
      tmem_ld_x32(tmem + lane_base + C::kS + 32, sr + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(u));
      float raw[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) raw[j] = __uint_as_float(sr[j]);
      if (__any_sync(0xffffffffu, nvis < kTile)) {
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j >= nvis) raw[j] = -INFINITY;
      }
      float g[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = max3(raw[16 * k], raw[16 * k + 1], raw[16 * k + 2]);
#pragma unroll
        for (int j = 3; j < 15; j += 2) a = max3(a, raw[16 * k + j], raw[16 * k + j + 1]);
        g[k] = fmaxf(a, raw[16 * k + 15]);
      }
      const float c = fmaxf(fmaxf(g[0], g[1]), fmaxf(g[2], g[3])) * cs;  // tile max, log2 units
      const bool empty = (c == -INFINITY);
      const float mt = (c > m + kTau) ? c : m;  // candidate frame (lazy maximum)
      uint32_t pw[8];
      uint32_t sfw = 0x08080808u;  // 2^-6 where nothing is visible
      float ell = 0.f;             // l_t: exact sum of the quantized P of this row
      if (!empty) {
        // the four group scales, clamped at 2^-6 (code 8), converted and decoded in pairs
        float gs[4], scv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) gs[k] = ex2_approx(fmaf(g[k], cs, -mt)) * (1.f / 6.f);
        sfw = cvt_ue4m3x4_min(gs[0], gs[1], gs[2], gs[3], 8u);
        ue4m3x4_values(sfw, scv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float nb = -(mt + lg2_approx(scv[k]));
#pragma unroll
          for (int w = 0; w < 2; ++w) pw[2 * k + w] = encode8(raw + 16 * k + 8 * w, cs, nb);
          ell = fmaf((float)(code_sum2(pw[2 * k]) + code_sum2(pw[2 * k + 1])), 0.5f * scv[k], ell);
        }
      } else {
#pragma unroll
        for (int w = 0; w < 8; ++w) pw[w] = 0u;
      }
      // hot test: w_t * l_t (in the committed frame) > eps * lambda
      const bool lift = !empty && mt != m;
      const bool lifted = __any_sync(0xffffffffu, lift);
      const float thr = eps == 0.f ? -1.f : eps * lam;
      const float ellw = ell * wt;
      bool vote;
      if (!lifted) vote = valid && !empty && ellw > thr;
      else vote = valid && !empty && !eps_inf &&
                  ((m == -INFINITY) ? (eps == 0.f || ellw > 0.f) : (ellw * ex2_approx(mt - m) > thr));
      const uint32_t bal = __ballot_sync(0xffffffffu, vote);
      const bool hot_lo = (bal & 0x0000FFFFu) != 0, hot_hi = (bal & 0xFFFF0000u) != 0;
      const bool hot = lane < 16 ? hot_lo : hot_hi;
      if (!lifted) {
        if (!empty) {
          lam += ell;
          if (!hot) l += ell;
        }
      } else {
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
        if (__any_sync(0xffffffffu, rescale)) {
          // O must not be touched before PV(u, i-1) has landed
          if (!(ok = warp_wait(pv_done(u, (i - 1) & 1), ((i - 1) >> 1) & 1))) break;
          tc_fence_after();
          const float fr = rescale ? f : 1.f;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(tO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * fr);
            tmem_st_x16(tO + c0, o);
            tmem_st_x16(tO + c0 + 16, o + 16);
          }
          tmem_wait_st();
        }
      }
      // P buffer (u, i % 2) and its scales were last read by PV(u, i-2).  A hot group's
      // scales are zero.
      if (i >= 2 && !(ok = warp_wait(pv_done(u, i & 1), ((i - 2) >> 1) & 1))) break;
      const int pbuf = 2 * u + (i & 1);
      uint8_t* pbp = smem + C::kPOff + 4096 * pbuf + (r >> 3) * 256 + (r & 7) * 16;
      *reinterpret_cast<uint4*>(pbp) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(pbp + 128) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      // the row's four P scales go straight into its own TMEM lane: a 32x128b.warpx4
      // copy of the 512-byte scale atom would put row 32c + l at lane l, column c of
      // every lane quarter, and lane quarter qw's MMA rows read column qw, so this one
      // word is the one the PV product reads for this row
      tmem_st_x1(tmem + lane_base + C::kSFP + 4 * pbuf + qw, hot ? 0u : sfw);
      if (lane == 0) gbits[u][i & 1][qw] = ((uint32_t)hot_lo << (2 * qw)) | ((uint32_t)hot_hi << (2 * qw + 1));
      if (p.hot_mask && (lane == 0 || lane == 16) && hot) {
        const int gi = (blk * kBlockRows + 32 * qw + lane) / kGroupRows;
        if (gi < ngroups) atomicOr(&p.hot_mask[((size_t)bh * ngroups + gi) * nwords + t / 32], 1u << (t % 32));
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(u, i & 1));
    }
    // ---- epilogue: the pass-1 state (o scaled by s_v, frame m, cold sum l)
    if (ok && n > 0) ok = warp_wait(pv_done(u, (n - 1) & 1), ((n - 1) >> 1) & 1);
    tc_fence_after();
    if (ok && blk < nblk) {
      const float sv = p.s_v[bh];
      float* orow = p.state_o + ((size_t)bh * nblk * kBlockRows + P) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld_x32(tO + c0, o);
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
  if (warp == kMmaS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Shared memory of the three-block kernel when it also runs the K/V quantizer:
// enough for either role, and more than half an SM's so that one CTA takes a
// whole SM (its TMEM allocation is the SM's 512 columns).
template <int D, int U>
constexpr int multi_kv_smem() {
  constexpr int a = P1MCfg<D, U>::kSmem, b = P1MCfg<D, U>::kQuantGroups * quant_role_smem(D) + 128,
                half = 114 * 1024 + 1024;
  return a > b ? (a > half ? a : half) : (b > half ? b : half);
}

template <int D, int U>
cudaError_t launch_multi(const P1Params& prm, cudaStream_t st) {
  using C = P1MCfg<D, U>;
  const int n_p1 = prm.s.BH() * ((prm.s.nblk() + U - 1) / U);
  if (!prm.kv_ready) {
    cudaError_t e =
        cudaFuncSetAttribute(pass1_multi_kernel<D, U>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e) return e;
    pass1_multi_kernel<D, U><<<n_p1, C::kThreads, C::kSmem, st>>>(prm);
    return cudaGetLastError();
  }
  // With the K/V quantizer: one CTA per SM, the pass-1 CTAs and a quantizer CTA on
  // every other SM, launched cooperatively because the pass-1 CTAs wait for the
  // quantizer's flags (all CTAs resident at once, so every wait ends).
  const int smem = multi_kv_smem<D, U>();
  cudaError_t e = cudaFuncSetAttribute(pass1_multi_kernel<D, U>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  P1Params prm2 = prm;
  prm2.n_p1 = n_p1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pass1_multi_kernel<D, U>, prm2);
}

// Shared memory of the one-block kernel when it also runs the K/V quantizer:
// enough for either role, and more than half an SM's (one CTA per SM).
template <int D>
constexpr int single_kv_smem() {
  constexpr int a = P1Cfg<D>::kSmem, b = P1Cfg<D>::kQuantGroups * quant_role_smem(D, P1Cfg<D>::kQuantBufs) + 128,
                half = 114 * 1024 + 1024;
  return a > b ? (a > half ? a : half) : (b > half ? b : half);
}

template <int D, bool kOnesMma>
cudaError_t launch_dv(const P1Params& prm, cudaStream_t st) {
  const int n_p1 = prm.s.BH() * prm.s.nblk();
  if (!prm.kv_ready) {
    const int smem = P1Cfg<D>::kSmem;
    cudaError_t e =
        cudaFuncSetAttribute(pass1_kernel<D, kOnesMma>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e) return e;
    pass1_kernel<D, kOnesMma><<<n_p1, p1_threads<D>(), smem, st>>>(prm);
    return cudaGetLastError();
  }
  if (kOnesMma) return cudaErrorInvalidValue;
  // with the K/V quantizer: one CTA per SM, cooperative (see launch_multi)
  const int smem = single_kv_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(pass1_kernel<D, kOnesMma>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) || (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
  P1Params prm2 = prm;
  prm2.n_p1 = n_p1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(p1_threads<D>());
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pass1_kernel<D, kOnesMma>, prm2);
}

// rowsum_mma: the ones-MMA row sums (one-block kernel); the default sums each
// row's quantized P in registers.
template <int D>
cudaError_t launch_d(const P1Params& prm, bool wide, bool rowsum_mma, cudaStream_t st) {
  // the residual Q term lives in the one-block kernel with register row sums
  if (prm.q2_blob) return launch_dv<D, false>(prm, st);
  if (rowsum_mma) return launch_dv<D, true>(prm, st);
  if constexpr (D <= 128) {
    if (!wide) return launch_multi<D, kUnits>(prm, st);
  }
  return launch_dv<D, false>(prm, st);
}

template <int D>
bool single_quantizes_kv(const Shape& s) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  const int n_p1 = s.BH() * s.nblk();
  if (sms - n_p1 < 8) return false;
  if (cudaFuncSetAttribute(pass1_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, single_kv_smem<D>()) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pass1_kernel<D, false>, p1_threads<D>(), single_kv_smem<D>()) !=
          cudaSuccess)
    return false;
  return per_sm == 1;
}

template <int D>
bool multi_quantizes_kv(const Shape& s) {
  constexpr int U = kUnits;
  using C = P1MCfg<D, U>;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  const int n_p1 = s.BH() * ((s.nblk() + U - 1) / U);
  if (sms - n_p1 < 8) return false;
  if (cudaFuncSetAttribute(pass1_multi_kernel<D, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           multi_kv_smem<D, U>()) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pass1_multi_kernel<D, U>, C::kThreads,
                                                    multi_kv_smem<D, U>()) != cudaSuccess)
    return false;
  return per_sm == 1;
}

}  // namespace

bool pass1_quantizes_kv(const Shape& s, bool wide, bool q_residual, bool rowsum_mma) {
  // the same choice of kernel as launch_d; the wide form shares the GPU and the
  // ones-MMA form has no room, so neither hosts the quantizer
  if (wide || rowsum_mma) return false;
  const bool one_block = q_residual || s.d > 128;
  switch (s.d) {
    case 64: return one_block ? single_quantizes_kv<64>(s) : multi_quantizes_kv<64>(s);
    case 128: return one_block ? single_quantizes_kv<128>(s) : multi_quantizes_kv<128>(s);
    case 256: return single_quantizes_kv<256>(s);
  }
  return false;
}

#ifdef APA_TEST_HOOKS
// Test builds only: while switched on, pass 1 with the K/V quantizer in its launch
// waits on a flag that nothing sets, so that its bounded wait runs out and the
// kernel unwinds; the call then reports APA_ERR_DEVICE through apa_check_error.
__device__ uint32_t g_never_set;
bool g_test_stuck = false;
}  // namespace apa
extern "C" int apa_test_stuck_quantizer_flags(int on) {
  apa::g_test_stuck = on != 0;
  return 0;
}
namespace apa {
#endif

cudaError_t launch_pass1(const Shape& s, const Workspace& ws, float eps, uint32_t* hot_mask, bool wide, cudaStream_t st,
                         const KvSource* kv, bool rowsum_mma) {
  P1Params prm{};
  prm.s = s;
  prm.kv_blob = ws.kv_blob;
  prm.q_blob = ws.q_blob;
  prm.q2_blob = ws.q2_blob;
  prm.s_k = ws.s_k;
  prm.s_v = ws.s_v;
  prm.s_q = ws.s_q;
  prm.eps = eps;
  prm.state_o = ws.state_o;
  prm.state_ml = ws.state_ml;
  prm.hot_list = ws.hot_list;
  prm.hot_count = ws.hot_count;
  prm.hot_mask = hot_mask;
  prm.wv = ws.wv;
  if (kv) {
    prm.kv_ready = ws.kv_ready;
    prm.k_raw = static_cast<const uint16_t*>(kv->k);
    prm.v_raw = static_cast<const uint16_t*>(kv->v);
    prm.ws = ws;
    prm.lse_scales = kv->lse ? 1 : 0;
#ifdef APA_TEST_HOOKS
    void* never = nullptr;
    if (g_test_stuck && cudaGetSymbolAddress(&never, g_never_set) == cudaSuccess)
      prm.test_never = static_cast<const uint32_t*>(never);
#endif
  }
  prm.err = device_error_word();
  switch (s.d) {
    case 64: return launch_d<64>(prm, wide, rowsum_mma, st);
    case 128: return launch_d<128>(prm, wide, rowsum_mma, st);
    case 256: return launch_d<256>(prm, wide, rowsum_mma, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace apa
