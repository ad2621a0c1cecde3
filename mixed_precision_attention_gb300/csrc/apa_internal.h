// apa_internal.h -- layouts and launchers shared by the library's .cu files.
//
// Notation: G = Hq/Hkv query heads share one KV head; packed row p = pos*G + g
// of KV head h holds query head h*G + g at position pos (GQA packing, so one
// K/V tile serves all G heads); R = G*Nq packed rows; rows come in 128-row
// blocks (one tcgen05 M tile) made of eight 16-row groups (the hot-test
// granularity); keys come in 64-key tiles, T = ceil(Nkv/64).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstring>

namespace apa {

constexpr int kTile = 64;        // keys per tile
constexpr int kBlockRows = 128;  // packed rows per block (tcgen05 M)
constexpr int kGroupRows = 16;   // rows per hot-test group
constexpr float kTau = 4.0f;     // lazy-max threshold (log2 units)
constexpr float kColdOffset = 32.0f;  // a hot tile lifts the frame to at most c - 32
constexpr float kLog2e = 1.4426950408889634f;

struct Shape {
  int B, Hq, Hkv, Nq, Nkv, d, causal;
  // Paged K/V (null: contiguous [B][Hkv][Nkv][d]): a pool of num_pages pages of
  // kTile keys, [page][Hkv][kTile][d], and a block table [B][max_pages] whose
  // entry t is the page holding keys kTile*t .. kTile*t + kTile-1 of sequence b.
  const int32_t* pages = nullptr;
  int max_pages = 0, num_pages = 0;
  __host__ __device__ int G() const { return Hq / Hkv; }
  __host__ __device__ int R() const { return G() * Nq; }
  __host__ __device__ int T() const { return (Nkv + kTile - 1) / kTile; }
  __host__ __device__ int nblk() const { return (R() + kBlockRows - 1) / kBlockRows; }
  __host__ __device__ int ngroups() const { return (R() + kGroupRows - 1) / kGroupRows; }
  __host__ __device__ int off() const { return Nkv - Nq; }
  __host__ __device__ int BH() const { return B * Hkv; }
};

// ------------------------------------------------------------------ NVFP4 tile blob
// One blob per (b, KV head, 64-key tile), in the exact shared-memory image the
// pass-1 MMAs read, so one bulk copy brings a tile in:
//   [0, 32d)        K codes:   B operand of S = Q K^T (N = 64 keys, K = d),
//                              canonical no-swizzle core matrices (8 rows x 16 B),
//                              LBO 128 B (along K), SBO 4d B (8-key groups);
//   [32d, 64d)      V^T codes: B operand of O += P V (N = d channels, K = 64 keys),
//                              LBO 128 B, SBO 256 B;
//   [64d, +ksf)     K scales: per pair of 64-channel k-blocks one 512-B chunk of
//                   32 rows x 16 B; row l = [key l kb0][key l+32 kb0][key l kb1][key l+32 kb1]
//                   (4 UE4M3 bytes each, one per 16 channels), copied to TMEM with
//                   tcgen05.cp 32x128b.warpx4 (k-block kb at column 4*(kb/2) + 2*(kb%2));
//   [.., +vsf)      V scales: per 128 channels one 512-B atom, byte (c%32)*16 + (c/32)*4 + kb16.
// E2M1 codes are packed two per byte, the lower index in the low nibble.
__host__ __device__ constexpr int sf_chunks(int d) { return (d + 127) / 128; }
__host__ __device__ constexpr int blob_kcodes(int) { return 0; }
__host__ __device__ constexpr int blob_vcodes(int d) { return 32 * d; }
__host__ __device__ constexpr int blob_ksf(int d) { return 64 * d; }
__host__ __device__ constexpr int blob_vsf(int d) { return 64 * d + 512 * sf_chunks(d); }
__host__ __device__ constexpr int blob_bytes(int d) { return 64 * d + 1024 * sf_chunks(d); }
// Q blob per 128-row block: codes (A operand, M = 128, K = d; LBO 128, SBO 4d) then
// one 512-B scale atom per 64-channel k-block (row p: byte (p%32)*16 + (p/32)*4 + kb16).
__host__ __device__ constexpr int qblob_sf(int d) { return 64 * d; }
__host__ __device__ constexpr int qblob_bytes(int d) { return 64 * d + 512 * (d / 64); }

// byte offset of the 8 code bytes of (row n, 16-element block cb) in a K-major
// no-swizzle operand whose rows hold `kbytes` bytes (K/2)
__host__ __device__ inline int fp4_kmajor_off(int n, int cb, int kbytes) {
  return (n >> 3) * (kbytes * 8) + (cb >> 1) * 128 + (n & 7) * 16 + 8 * (cb & 1);
}
// byte offset of the scale of (row r < 128, k16 block) in a 512-B scale atom
__host__ __device__ inline int sf_atom_off(int r, int k16) { return (r & 31) * 16 + (r >> 5) * 4 + k16; }

// ------------------------------------------------------------------ workspace
struct Workspace {
  // quantizer
  float* ksum;        // [BH][T][d] FP32 per-tile key sums
  uint32_t* kmin;     // [BH][d] orderable-encoded per-channel min of K
  uint32_t* kmax;     // [BH][d]
  uint32_t* vamax;    // [BH] max |v| (float bits)
  uint32_t* qamax;    // [B*Hq] max |q| (float bits)
  uint32_t* kcamax;   // [BH] max |k - mu| (float bits)
  float* mu;          // [BH][d]
  float* s_k;         // [BH]
  float* s_v;         // [BH]
  float* s_q;         // [B*Hq]
  uint8_t* kv_blob;   // [BH][T][blob_bytes(d)]
  uint8_t* q_blob;    // [BH][nblk][qblob_bytes(d)]
  uint8_t* q2_blob;   // [BH][nblk][qblob_bytes(d)] the FP4 residual term of Q, or null
  uint16_t* v16;      // [BH][Nkv][d] FP16 copy of V / v16_scale(max |v|) for pass 2, or null
  float* wv;          // [BH][T] largest key value norm of each tile, then (after the key
                      // mean) the tile's hot-test weight; null unless value-weighted
  float* vtsum;       // [BH][T] FP32 sum of the tile's key value norms (with wv)
  uint32_t* kv_ready; // [BH*T + 1]: per tile 1 once its blob is written by the K/V
                      // quantizer inside the pass-1 launch; the last word is that
                      // quantizer's ticket counter
  // pass 1 -> pass 2
  float* state_o;     // [BH][nblk*128][d]: pass-1 o (scaled by s_v)
  float2* state_ml;   // [BH][nblk*128]: pass-1 frame m and cold sum l
  uint32_t* hot_list; // [BH*nblk][T]: tile | group mask << 16
  uint32_t* hot_count;// [BH*nblk]
  uint32_t* p2_order; // [BH*nblk]: pass-2 work items (bh * nblk + blk), longest hot list first
  // d = 256: the parts of a split pass-2 walk (exact_split(s) > 1 in the all-exact
  // mode, apa_split(s) > 1 in APA mode), else null
  float* part_o;      // [BH*nblk*nsplit][128][d]
  float2* part_ml;    // [BH*nblk*nsplit][128]
  float* part_qmu;    // [BH*nblk][128], APA mode: each row's LSE term q.mu / sqrt(d)
};
// apa_mode false (eps = 0): only the FP16 copy of V and the head maxima of V.
// flags: APA_FLAG_* of apa.h (APA_FLAG_Q_RESIDUAL adds the residual Q blob)
size_t workspace_layout(const Shape& s, bool apa_mode, Workspace* ws, void* base, unsigned flags = 0);
// The parts into which the all-exact pass 2 splits each block's walk: at d = 256
// (the one-group kernel, one CTA per 128-row block) with few blocks per (b, KV head)
// and a long walk, one part per 1024 tiles, at most 4.  It depends on the
// per-(b, KV head) shape only, so the sub-problems of the host entry point split
// the same way as the whole call.
inline int exact_split(const Shape& s) {
  if (s.d <= 128 || s.nblk() > 4) return 1;
  const int k = s.T() / 1024;
  return k < 1 ? 1 : (k > 4 ? 4 : k);
}
// The same for the APA-mode pass 2, whose walk is the block's hot list: a few
// percent of the tiles, but the longest lists still set its time when there are
// few blocks.  One part per 512 tiles of the context, at most 4.
inline int apa_split(const Shape& s) {
  if (s.d <= 128 || s.nblk() > 4) return 1;
  const int k = s.T() / 512;
  return k < 1 ? 1 : (k > 4 ? 4 : k);
}

// Power-of-two divisor that brings a head's V into FP16 range: 1 when max |v| is
// at most 2^15, else 2^(e - 14) for max |v| in [2^e, 2^(e+1)).  Dividing by it is
// exact, so the FP16 copy holds every bf16 value of V exactly except those below
// 2^-17 times the divisor (FP16 subnormals), which round to a multiple of 2^-24.
__host__ __device__ inline float v16_scale(float vamax) {
  int e = 0;
  if (vamax > 32768.f) {
    uint32_t bits;
    memcpy(&bits, &vamax, 4);
    e = (int)((bits >> 23) & 0xFF) - 127 - 14;
  }
  uint32_t sb = (uint32_t)(127 + e) << 23;
  float sc;
  memcpy(&sc, &sb, 4);
  return sc;
}

int* device_error_word();  // library-wide device error word (set by bounded waits)

#ifdef __CUDACC__
// The page of key tile t of head (b, h) in a paged K/V pool; an entry outside the
// pool reads page 0 and records APA_DEVERR_BOUNDS (2) in *err.
__device__ __forceinline__ int kv_page(const Shape& s, int b, int t, int* err) {
  int pg = s.pages[(size_t)b * s.max_pages + t];
  if (pg < 0 || pg >= s.num_pages) {
    if (err) atomicCAS(err, 0, 2);
    pg = 0;
  }
  return pg;
}
// Element offset, in K or V, of the first key of tile t of head bh.
__device__ __forceinline__ size_t kv_tile_offset(const Shape& s, int bh, int t, int* err) {
  if (!s.pages) return ((size_t)bh * s.Nkv + (size_t)t * kTile) * s.d;
  const int b = bh / s.Hkv, h = bh % s.Hkv;
  return (((size_t)kv_page(s, b, t, err) * s.Hkv + h) * kTile) * s.d;
}
#endif


// ------------------------------------------------------------------ launchers
// lse: least-squared-error block scales (APA_FLAG_LSE_SCALES) instead of the nearest ones.
// kv_in_pass1: the K/V tiles are left to the quantizer inside the pass-1 launch
// (launch_pass1 with a KvSource): this call then runs the statistics and the Q
// blocks (which also publish the K/V head scales) and clears ws.kv_ready.
cudaError_t launch_quantize(const Shape& s, const void* q, const void* k, const void* v, const Workspace& ws,
                            bool do_q, bool do_kv, cudaStream_t st, bool lse = false, bool kv_in_pass1 = false);
// The raw K and V for the K/V quantizer that runs inside the pass-1 launch.
struct KvSource {
  const void* k;
  const void* v;
  bool lse;
};
// Whether the pass-1 launch for this problem can quantize the K/V tiles itself
// (the three-block kernel, with at least 8 SMs left over for the quantizer).
bool pass1_quantizes_kv(const Shape& s, bool wide, bool q_residual, bool rowsum_mma);
// wide: one 128-row block per CTA (three times the CTAs, each on its own SM when
// the GPU is otherwise idle, so a single problem finishes sooner) instead of
// three blocks of one KV head per CTA (the faster choice for a full GPU).
// kv: quantize the K/V tiles inside this launch (pass1_quantizes_kv must hold).
// rowsum_mma: tile row sums from an MMA against an E2M1 ones tile (APA_FLAG_ROWSUM_MMA).
cudaError_t launch_pass1(const Shape& s, const Workspace& ws, float eps, uint32_t* hot_mask, bool wide,
                         cudaStream_t st, const KvSource* kv = nullptr, bool rowsum_mma = false);
cudaError_t launch_pass2(const Shape& s, const void* q, const void* k, const void* v, const Workspace* ws,
                         float* out, float* lse, cudaStream_t st);
// The all-exact path's FP16 copy of V (ws.v16, with the head maxima in ws.vamax):
// V divided by v16_scale(max |v|) per head, the copy the quantizer writes in APA mode.
cudaError_t launch_v16(const Shape& s, const void* v, const Workspace& ws, cudaStream_t st);
cudaError_t launch_visible_mask(const Shape& s, uint32_t* hot_mask, cudaStream_t st);
cudaError_t launch_pass2_order(const Shape& s, const Workspace& ws, cudaStream_t st);

}  // namespace apa
