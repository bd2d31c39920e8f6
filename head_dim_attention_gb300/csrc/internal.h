// Host/device parameter blocks and launcher declarations shared between the
// C-ABI layer (api.cu) and the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ffpa {

// Device status word values (written with atomicCAS so the first error wins).
enum : uint32_t {
  FFPA_DEV_OK = 0,
  FFPA_DEV_TIMEOUT = 1,
  FFPA_DEV_LAYOUT = 2,  // dynamic shared memory not on the boundary a kernel's layout needs
};

constexpr int kTileRows = 128;  // query/key rows per tile (the MMA M)
constexpr int kChunk = 64;      // D columns per chunk (one 128-byte swizzled row)
constexpr int kChunkBytes = kTileRows * kChunk * 2;  // 16 KB

// Forward, fused tcgen05 path.
struct FwdParams {
  void* out;
  float* lse;         // nullable, contiguous [B, Hq, Nq]
  const float* bias;  // nullable
  const void* q;      // read directly (not through TMA) by the full-D pair kernel
  int64_t q_sb, q_sh, q_sn;
  int64_t o_sb, o_sh, o_sn;
  int64_t bias_sb, bias_sh, bias_sq, bias_sk;
  int bias_vec;       // bias rows contiguous along the keys and 16-byte aligned: 4 keys per load
  int B, Hq, Hkv, Nq, Nkv, D;
  int group;          // Hq / Hkv
  int causal;
  float scale_log2;   // scale * log2(e)
  int n_chunks;       // D / 64
  int stages;         // ring slots
  int slot_chunks;    // 64-column chunk tiles per ring slot (1 or 2), loaded under one barrier phase
  int q_tiles;        // ceil(Nq / 128)
  uint32_t* status;   // device status word
  // split over the keys (short query sets): each CTA pair takes kv_split_tiles
  // key tiles and writes an unnormalised partial O and its (max, sum) for the
  // decode path's combine kernel; part_o == nullptr: no split
  int kv_splits, kv_split_tiles;
  float* part_o;      // [B, Hq, Nq, kv_splits, D] fp32
  float* part_ml;     // [B, Hq, Nq, kv_splits, 2] fp32 (max, sum), log2 domain
  // dropout (philox.cuh): on when `dropout` is set; keep threshold, seed words,
  // stream offset and the multiplier 1 / (1 - p) of kept probabilities
  int dropout;
  uint32_t drop_t, drop_seed_lo, drop_seed_hi, drop_off;
  float drop_scale;
};

struct FwdMaps {
  CUtensorMap q, k, v;  // 4-D {D, N, H, B}, box {64, 128, 1, 1}, 128-byte swizzle
  CUtensorMap k_half;   // K with box {64, 64, 1, 1}: one CTA's half of a key tile in the CTA-pair kernels
  CUtensorMap q_half;   // Q with box {64, 64, 1, 1}: one CTA's 64 query rows in the full-D pair kernel
};

// Decode (small Nq) path.
struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  const float* bias;
  int64_t q_sb, q_sh, q_sn;
  int64_t k_sb, k_sh, k_sn;
  int64_t v_sb, v_sh, v_sn;
  int64_t o_sb, o_sh, o_sn;
  int64_t bias_sb, bias_sh, bias_sq, bias_sk;
  int B, Hq, Hkv, Nq, Nkv, D;
  int group;
  int causal;
  float scale_log2;
  int heads_per_cta;  // query heads (of one kv head) per split CTA: 1 or the GQA group
  int split_len;      // keys per split
  int n_splits;
  float* part_o;      // [B, Hq, Nq, n_splits, D] fp32 scratch
  float* part_ml;     // [B, Hq, Nq, n_splits, 2] fp32 scratch (max, sum), log2 domain
  uint32_t* status;   // device status word (bounded waits of the streaming kernel)
};

// Backward.
struct BwdParams {
  const void* out;
  const void* dout;
  const float* lse;   // [B, Hq, Nq] natural log
  float* delta;       // [B, Hq, Nq] scratch
  float* lse2;        // [B, Hq, Nq] scratch: lse in log2 units
  const float* bias;
  void* dq;
  void* dk;
  void* dv;
  const void* q;      // read directly (not through TMA) by the dQ and fused dK/dV kernels
  const void* k;
  const void* v;
  int64_t q_sb, q_sh, q_sn;
  int64_t k_sb, k_sh, k_sn;
  int64_t v_sb, v_sh, v_sn;
  int64_t o_sb, o_sh, o_sn;
  int64_t do_sb, do_sh, do_sn;
  int64_t dq_sb, dq_sh, dq_sn;
  int64_t dk_sb, dk_sh, dk_sn;
  int64_t dv_sb, dv_sh, dv_sn;
  int64_t bias_sb, bias_sh, bias_sq, bias_sk;
  int B, Hq, Hkv, Nq, Nkv, D;
  int group;
  int causal;
  float scale;
  float scale_log2;
  int n_chunks;
  int stages;         // ring slots
  int slot_chunks;    // 16 KB tiles per ring slot (1 or 2), loaded under one barrier phase
  int q_tiles, kv_tiles;
  uint32_t* status;
  // dropout, as in FwdParams
  int dropout;
  uint32_t drop_t, drop_seed_lo, drop_seed_hi, drop_off;
  float drop_scale;
};

struct BwdMaps {
  CUtensorMap q, k, v, dout;                  // box {64, 128, 1, 1}
  CUtensorMap q_half, k_half, v_half, dout_half;  // box {64, 64, 1, 1}: one CTA's half of a column tile (CTA pair)
};

bool dtype_is_bf16(int dtype);

cudaError_t launch_fwd_main(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s);
// Full-D CTA-pair forward (fwd_fulld.cu): D = 512, one pair holds all of O.
bool fwd_fulld_supported(const FwdParams& p);
// Key splits (1: none) for a short query set on `sms` SMs, and key tiles per split.
int fwd_fulld_kv_splits(const FwdParams& p, int sms, int* tiles_per_split);
cudaError_t launch_fwd_fulld(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s);
// Forward for D = 704 .. 1024 on clusters of two CTA pairs (fwd_xch.cu): one
// pair computes S and P, the other holds all of O; no dropout, no key split.
bool fwd_xch_supported(const FwdParams& p);
cudaError_t launch_fwd_xch(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s);
cudaError_t launch_fwd_decode(const DecodeParams& p, bool bf16, cudaStream_t s);
// The decode path's merge of per-split partials (part_o, part_ml) into out and
// lse; also merges the key splits of the full-D forward for short query sets.
cudaError_t launch_decode_combine(const DecodeParams& p, bool bf16, cudaStream_t s);
int decode_heads_per_cta(int group, int Nq, int D);
// Same kernels, partials in the library's fixed device array (no allocation).
cudaError_t launch_fwd_decode_noalloc(const DecodeParams& p, bool bf16, cudaStream_t s);
size_t decode_scratch_bytes(const DecodeParams& p);
size_t decode_noalloc_capacity_bytes();
cudaError_t launch_bwd(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s);
// Full-D CTA-pair dQ kernel (bwd_dq.cu): D = 320 .. 512; the preprocess runs first.
bool bwd_dq_supported(const BwdParams& p);
cudaError_t launch_bwd_dq(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s);
// Exchange kernel on clusters of two CTA pairs (bwd_xch.cu): its fused dK/dV
// mode (D = 320 .. 1024) and its dQ mode (D = 576 .. 1024), after the preprocess.
bool bwd_xch_dkv_supported(const BwdParams& p);
bool bwd_xch_dq_supported(const BwdParams& p);
cudaError_t launch_bwd_xch_dkv(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_xch_dq(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s);

uint32_t* device_status_word();  // per current device

// Measurement hook (ffpa_set_timing_events): record the caller's next event
// on `s`; a no-op unless the calling thread registered events.
void timing_mark(cudaStream_t s);

}  // namespace ffpa
