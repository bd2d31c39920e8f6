// C ABI: argument validation, TMA descriptor encoding and dispatch.
// Every check runs on the host before anything is enqueued; on failure the
// call returns a status and launches nothing.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "ffpa.h"
#include "internal.h"
#include "ptx.cuh"

namespace ffpa {

// Per-device status word, set by kernels whose bounded waits expire.
__device__ uint32_t g_status_word;

uint32_t* device_status_word() {
  static std::mutex mu;
  static uint32_t* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint32_t*>(ptr);
  }
  return cache[dev];
}

bool dtype_is_bf16(int dtype) { return dtype == FFPA_BF16; }

namespace {
struct TimingHook {
  cudaEvent_t ev[8];
  int n = 0;
  int next = 0;
};
thread_local TimingHook g_hook;
void timing_begin() { g_hook.next = 0; }
}  // namespace

void timing_mark(cudaStream_t s) {
  if (g_hook.next < g_hook.n) cudaEventRecord(g_hook.ev[g_hook.next++], s);
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct Shape4 {
  int64_t B, H, N, D;
};

bool is_half_dtype(int dt) { return dt == FFPA_F16 || dt == FFPA_BF16; }

// Validate one [B, H, N, D] half-precision tensor.
int check_bhnd(const ffpa_tensor_t* t, int dtype, const Shape4& want) {
  if (!t || !t->data || t->reserved != 0) return FFPA_ERR_INVALID_ARG;
  if (t->dtype != dtype) return is_half_dtype(t->dtype) ? FFPA_ERR_INVALID_ARG : FFPA_ERR_UNSUPPORTED;
  if (t->shape[0] != want.B || t->shape[1] != want.H || t->shape[2] != want.N || t->shape[3] != want.D)
    return FFPA_ERR_INVALID_ARG;
  if (t->stride[3] != 1) return FFPA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return FFPA_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i) {
    if (t->shape[i] > 1 && (t->stride[i] <= 0 || t->stride[i] % 8 != 0)) return FFPA_ERR_ALIGNMENT;
  }
  return FFPA_OK;
}

// Natural strides for size-1 dims so the TMA descriptor sees a well-formed map.
void tma_strides(const ffpa_tensor_t* t, int64_t out[3]) {
  // out[0] = row stride, out[1] = head stride, out[2] = batch stride (elements)
  int64_t sn = t->shape[2] > 1 ? t->stride[2] : t->shape[3];
  int64_t sh = t->shape[1] > 1 ? t->stride[1] : sn * t->shape[2];
  int64_t sb = t->shape[0] > 1 ? t->stride[0] : sh * t->shape[1];
  out[0] = sn;
  out[1] = sh;
  out[2] = sb;
}

int encode_map(CUtensorMap* m, const ffpa_tensor_t* t, int box_rows = kTileRows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FFPA_ERR_CUDA;
  int64_t st[3];
  tma_strides(t, st);
  const cuuint64_t dims[4] = {(cuuint64_t)t->shape[3], (cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1],
                              (cuuint64_t)t->shape[0]};
  const cuuint64_t strides[3] = {(cuuint64_t)st[0] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[2] * 2};
  const cuuint32_t box[4] = {(cuuint32_t)kChunk, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      t->dtype == FFPA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(m, dt, 4, t->data, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FFPA_OK : FFPA_ERR_CUDA;
}

struct Common {
  int64_t B, Hq, Hkv, Nq, Nkv, D;
  int dtype;
};

int check_common(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                 const ffpa_tensor_t* bias, float scale, Common* c) {
  if (!q || !k || !v) return FFPA_ERR_INVALID_ARG;
  if (!is_half_dtype(q->dtype)) return FFPA_ERR_UNSUPPORTED;
  c->dtype = q->dtype;
  c->B = q->shape[0];
  c->Hq = q->shape[1];
  c->Nq = q->shape[2];
  c->D = q->shape[3];
  c->Hkv = k->shape[1];
  c->Nkv = k->shape[2];
  if (c->B < 1 || c->Hq < 1 || c->Hkv < 1 || c->Nq < 1 || c->Nkv < 1 || c->D < 1) return FFPA_ERR_INVALID_ARG;
  if (c->B > 65535 || c->Hq > 65535 || c->Nq > (1ll << 30) || c->Nkv > (1ll << 30)) return FFPA_ERR_UNSUPPORTED;
  if (c->Hq % c->Hkv != 0) return FFPA_ERR_INVALID_ARG;
  if (c->D % 64 != 0 || c->D < 64 || c->D > 1024) return FFPA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FFPA_ERR_INVALID_ARG;
  int rc = check_bhnd(q, c->dtype, {c->B, c->Hq, c->Nq, c->D});
  if (rc) return rc;
  rc = check_bhnd(k, c->dtype, {c->B, c->Hkv, c->Nkv, c->D});
  if (rc) return rc;
  rc = check_bhnd(v, c->dtype, {c->B, c->Hkv, c->Nkv, c->D});
  if (rc) return rc;
  if (bias) {
    if (!bias->data || bias->reserved != 0) return FFPA_ERR_INVALID_ARG;
    if (bias->dtype != FFPA_F32) return FFPA_ERR_UNSUPPORTED;
    const int64_t* s = bias->shape;
    if (!(s[0] == 1 || s[0] == c->B) || !(s[1] == 1 || s[1] == c->Hq) || !(s[2] == 1 || s[2] == c->Nq) ||
        s[3] != c->Nkv)
      return FFPA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(bias->data) % 4 != 0) return FFPA_ERR_ALIGNMENT;
  }
  return FFPA_OK;
}

int check_lse(const ffpa_tensor_t* lse, const Common& c) {
  if (!lse->data || lse->reserved != 0) return FFPA_ERR_INVALID_ARG;
  if (lse->dtype != FFPA_F32) return FFPA_ERR_UNSUPPORTED;
  if (lse->shape[0] != c.B || lse->shape[1] != c.Hq || lse->shape[2] != c.Nq || lse->shape[3] != 1)
    return FFPA_ERR_INVALID_ARG;
  // contiguous [B, Hq, Nq]
  if ((c.Nq > 1 && lse->stride[2] != 1) || (c.Hq > 1 && lse->stride[1] != c.Nq) ||
      (c.B > 1 && lse->stride[0] != c.Hq * c.Nq))
    return FFPA_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(lse->data) % 4 != 0) return FFPA_ERR_ALIGNMENT;
  return FFPA_OK;
}

void bias_strides(const ffpa_tensor_t* bias, int64_t* sb, int64_t* sh, int64_t* sq, int64_t* sk) {
  if (!bias) {
    *sb = *sh = *sq = *sk = 0;
    return;
  }
  *sb = bias->shape[0] > 1 ? bias->stride[0] : 0;
  *sh = bias->shape[1] > 1 ? bias->stride[1] : 0;
  *sq = bias->shape[2] > 1 ? bias->stride[2] : 0;
  *sk = bias->stride[3];
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA; }

constexpr int kDecodeMaxRows = 16;

// Keys per decode slice: the multiple of 16 in [128, 256] for which the
// decode CTAs (one per batch, group of query heads sharing a kv head, and
// slice; two fit on an SM) fill their last wave best on the current device;
// `Hq` counts those groups.  Ties go to the longer slice.
// Slices of at least 128 keys keep a call's partials within what 128-key
// slices would take (the no-allocation entry point's capacity check).
// Stream-ordered scratch (backward Delta and lse2, decode and key-split
// partials) comes from a memory pool the library creates per device and whose
// release threshold keeps freed blocks reserved: after the first call of a
// size, an allocation reuses them instead of mapping new memory, which with a
// default pool (threshold 0) happened on every call and left the GPU idle for
// tens of microseconds while the host mapped it.
cudaError_t scratch_alloc(void** ptr, size_t bytes, cudaStream_t st) {
  static std::mutex mu;
  static cudaMemPool_t pools[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      cudaMemPool_t created;
      if ((e = cudaMemPoolCreate(&created, &props)) != cudaSuccess) return e;
      uint64_t keep = UINT64_MAX;
      if ((e = cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) return e;
      pools[dev] = created;
    }
    pool = pools[dev];
  }
  return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

// SMs of the current device (cached per device; 0 if unknown).
int device_sm_count() {
  static std::mutex mu;
  static int sms_cache[64] = {};
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (!sms_cache[dev]) {
      int v = 0;
      if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) sms_cache[dev] = v;
    }
    sms = sms_cache[dev];
  }
  return sms;
}

int decode_split_len(int64_t B, int64_t Hq, int64_t Nkv) {
  const int sms = device_sm_count();
  if (sms <= 0) return 128;
  const int64_t slots = 2 * static_cast<int64_t>(sms);
  int best = 128;
  double best_fill = -1.0;
  for (int L = 256; L >= 128; L -= 16) {
    const int64_t ctas = B * Hq * ((Nkv + L - 1) / L);
    const int64_t waves = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = L;
    }
  }
  return best;
}
constexpr float kLog2e = 1.4426950408889634f;

}  // namespace
}  // namespace ffpa

using namespace ffpa;

namespace {

// Dropout arguments as the entry points take them; p == 0 is no dropout.
struct DropArgs {
  double p;
  uint64_t seed;
  uint32_t offset;
};

// Checks p (0 <= p < 1) and derives the kernels' parameters: the 16-bit keep
// threshold round(p * 65536) (at most 65535) and the multiplier 1 / (1 - p).
int drop_params(const DropArgs* d, int* on, uint32_t* t, uint32_t* seed_lo, uint32_t* seed_hi, uint32_t* off,
                float* scale) {
  *on = 0;
  *t = 0;
  *seed_lo = *seed_hi = *off = 0;
  *scale = 1.f;
  if (!d) return FFPA_OK;
  if (!(d->p >= 0.0 && d->p < 1.0)) return FFPA_ERR_INVALID_ARG;
  if (d->p == 0.0) return FFPA_OK;
  *on = 1;
  *t = static_cast<uint32_t>(std::min(65535.0, std::floor(d->p * 65536.0 + 0.5)));
  *seed_lo = static_cast<uint32_t>(d->seed);
  *seed_hi = static_cast<uint32_t>(d->seed >> 32);
  *off = d->offset;
  *scale = static_cast<float>(1.0 / (1.0 - d->p));
  return FFPA_OK;
}

int fwd_impl(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v, const ffpa_tensor_t* bias,
             int causal, float scale, const DropArgs* drop, const ffpa_tensor_t* out, const ffpa_tensor_t* lse,
             ffpa_stream_t stream) {
  Common c;
  int rc = check_common(q, k, v, bias, scale, &c);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FFPA_ERR_INVALID_ARG;
  int dropout;
  uint32_t drop_t, seed_lo, seed_hi, drop_off;
  float drop_scale;
  if ((rc = drop_params(drop, &dropout, &drop_t, &seed_lo, &seed_hi, &drop_off, &drop_scale))) return rc;
  if (dropout && c.D < 320) return FFPA_ERR_UNSUPPORTED;  // dropout: the D = 320 .. 1024 kernels
  rc = check_bhnd(out, c.dtype, {c.B, c.Hq, c.Nq, c.D});
  if (rc) return rc;
  if (lse && (rc = check_lse(lse, c))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = device_status_word();
  if (!status) return FFPA_ERR_CUDA;
  const bool bf16 = dtype_is_bf16(c.dtype);
  int64_t bsb, bsh, bsq, bsk;
  bias_strides(bias, &bsb, &bsh, &bsq, &bsk);
  timing_begin();

  if (c.Nq <= kDecodeMaxRows && !dropout) {
    DecodeParams p = {};
    p.q = q->data;
    p.k = k->data;
    p.v = v->data;
    p.out = out->data;
    p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
    p.bias = bias ? static_cast<const float*>(bias->data) : nullptr;
    p.q_sb = q->stride[0]; p.q_sh = q->stride[1]; p.q_sn = q->stride[2];
    p.k_sb = k->stride[0]; p.k_sh = k->stride[1]; p.k_sn = k->stride[2];
    p.v_sb = v->stride[0]; p.v_sh = v->stride[1]; p.v_sn = v->stride[2];
    p.o_sb = out->stride[0]; p.o_sh = out->stride[1]; p.o_sn = out->stride[2];
    p.bias_sb = bsb; p.bias_sh = bsh; p.bias_sq = bsq; p.bias_sk = bsk;
    p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.Nq = (int)c.Nq; p.Nkv = (int)c.Nkv; p.D = (int)c.D;
    p.group = (int)(c.Hq / c.Hkv);
    p.causal = causal;
    p.scale_log2 = scale * kLog2e;
    p.heads_per_cta = decode_heads_per_cta(p.group, p.Nq, p.D);
    p.split_len = decode_split_len(c.B, c.Hq / p.heads_per_cta, c.Nkv);
    p.n_splits = (int)((c.Nkv + p.split_len - 1) / p.split_len);
    p.status = status;
    const size_t n_rows = (size_t)c.B * c.Hq * c.Nq * p.n_splits;
    void* scratch = nullptr;
    const size_t o_bytes = n_rows * c.D * sizeof(float), ml_bytes = n_rows * 2 * sizeof(float);
    if (scratch_alloc(&scratch, o_bytes + ml_bytes, st) != cudaSuccess) return FFPA_ERR_CUDA;
    p.part_o = static_cast<float*>(scratch);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes);
    cudaError_t e = launch_fwd_decode(p, bf16, st);
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return cuda_rc(e != cudaSuccess ? e : e2);
  }

  FwdParams p = {};
  p.out = out->data;
  p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
  p.bias = bias ? static_cast<const float*>(bias->data) : nullptr;
  p.q = q->data;
  p.q_sb = q->stride[0]; p.q_sh = q->stride[1]; p.q_sn = q->stride[2];
  p.o_sb = out->stride[0]; p.o_sh = out->stride[1]; p.o_sn = out->stride[2];
  p.bias_sb = bsb; p.bias_sh = bsh; p.bias_sq = bsq; p.bias_sk = bsk;
  p.bias_vec = bias && bsk == 1 && reinterpret_cast<uintptr_t>(bias->data) % 16 == 0 && bsb % 4 == 0 &&
               bsh % 4 == 0 && bsq % 4 == 0;
  p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.Nq = (int)c.Nq; p.Nkv = (int)c.Nkv; p.D = (int)c.D;
  p.group = (int)(c.Hq / c.Hkv);
  p.causal = causal;
  p.scale_log2 = scale * kLog2e;
  p.n_chunks = (int)(c.D / kChunk);
  p.q_tiles = (int)((c.Nq + kTileRows - 1) / kTileRows);
  p.status = status;
  p.dropout = dropout;
  p.drop_t = drop_t; p.drop_seed_lo = seed_lo; p.drop_seed_hi = seed_hi; p.drop_off = drop_off;
  p.drop_scale = drop_scale;
  FwdMaps m;
  if ((rc = encode_map(&m.q, q)) || (rc = encode_map(&m.k, k)) || (rc = encode_map(&m.v, v)) ||
      (rc = encode_map(&m.k_half, k, kTileRows / 2)) || (rc = encode_map(&m.q_half, q, kTileRows / 2)))
    return rc;
  int per = 0;
  const int splits = fwd_fulld_supported(p) ? fwd_fulld_kv_splits(p, device_sm_count(), &per) : 1;
  if (splits > 1) {
    // a short query set: the key splits write partials, the combine merges them
    const size_t n_rows = (size_t)c.B * c.Hq * c.Nq * splits;
    const size_t o_bytes = n_rows * c.D * sizeof(float), ml_bytes = n_rows * 2 * sizeof(float);
    void* scratch = nullptr;
    if (scratch_alloc(&scratch, o_bytes + ml_bytes, st) != cudaSuccess) return FFPA_ERR_CUDA;
    p.kv_splits = splits;
    p.kv_split_tiles = per;
    p.part_o = static_cast<float*>(scratch);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) + o_bytes);
    cudaError_t e = launch_fwd_main(p, m, bf16, st);
    if (e == cudaSuccess) {
      DecodeParams dp = {};
      dp.out = out->data;
      dp.lse = p.lse;
      dp.o_sb = p.o_sb; dp.o_sh = p.o_sh; dp.o_sn = p.o_sn;
      dp.B = p.B; dp.Hq = p.Hq; dp.Hkv = p.Hkv; dp.Nq = p.Nq; dp.Nkv = p.Nkv; dp.D = p.D;
      dp.n_splits = splits;
      dp.part_o = p.part_o;
      dp.part_ml = p.part_ml;
      dp.status = status;
      e = launch_decode_combine(dp, bf16, st);
    }
    cudaError_t e2 = cudaFreeAsync(scratch, st);
    return cuda_rc(e != cudaSuccess ? e : e2);
  }
  return cuda_rc(launch_fwd_main(p, m, bf16, st));
}

int bwd_impl(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v, const ffpa_tensor_t* bias,
             int causal, float scale, const DropArgs* drop, const ffpa_tensor_t* out, const ffpa_tensor_t* lse,
             const ffpa_tensor_t* dout, const ffpa_tensor_t* dq, const ffpa_tensor_t* dk, const ffpa_tensor_t* dv,
             ffpa_stream_t stream) {
  Common c;
  int rc = check_common(q, k, v, bias, scale, &c);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FFPA_ERR_INVALID_ARG;
  int dropout;
  uint32_t drop_t, seed_lo, seed_hi, drop_off;
  float drop_scale;
  if ((rc = drop_params(drop, &dropout, &drop_t, &seed_lo, &seed_hi, &drop_off, &drop_scale))) return rc;
  if (dropout && c.D < 320) return FFPA_ERR_UNSUPPORTED;
  if ((rc = check_bhnd(out, c.dtype, {c.B, c.Hq, c.Nq, c.D}))) return rc;
  if ((rc = check_bhnd(dout, c.dtype, {c.B, c.Hq, c.Nq, c.D}))) return rc;
  if ((rc = check_bhnd(dq, c.dtype, {c.B, c.Hq, c.Nq, c.D}))) return rc;
  if ((rc = check_bhnd(dk, c.dtype, {c.B, c.Hkv, c.Nkv, c.D}))) return rc;
  if ((rc = check_bhnd(dv, c.dtype, {c.B, c.Hkv, c.Nkv, c.D}))) return rc;
  if (!lse) return FFPA_ERR_INVALID_ARG;
  if ((rc = check_lse(lse, c))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = device_status_word();
  if (!status) return FFPA_ERR_CUDA;
  int64_t bsb, bsh, bsq, bsk;
  bias_strides(bias, &bsb, &bsh, &bsq, &bsk);
  BwdParams p = {};
  p.out = out->data;
  p.dout = dout->data;
  p.lse = static_cast<const float*>(lse->data);
  p.bias = bias ? static_cast<const float*>(bias->data) : nullptr;
  p.dq = dq->data;
  p.dk = dk->data;
  p.dv = dv->data;
  p.q = q->data;
  p.k = k->data;
  p.v = v->data;
  p.q_sb = q->stride[0]; p.q_sh = q->stride[1]; p.q_sn = q->stride[2];
  p.k_sb = k->stride[0]; p.k_sh = k->stride[1]; p.k_sn = k->stride[2];
  p.v_sb = v->stride[0]; p.v_sh = v->stride[1]; p.v_sn = v->stride[2];
  p.o_sb = out->stride[0]; p.o_sh = out->stride[1]; p.o_sn = out->stride[2];
  p.do_sb = dout->stride[0]; p.do_sh = dout->stride[1]; p.do_sn = dout->stride[2];
  p.dq_sb = dq->stride[0]; p.dq_sh = dq->stride[1]; p.dq_sn = dq->stride[2];
  p.dk_sb = dk->stride[0]; p.dk_sh = dk->stride[1]; p.dk_sn = dk->stride[2];
  p.dv_sb = dv->stride[0]; p.dv_sh = dv->stride[1]; p.dv_sn = dv->stride[2];
  p.bias_sb = bsb; p.bias_sh = bsh; p.bias_sq = bsq; p.bias_sk = bsk;
  p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.Nq = (int)c.Nq; p.Nkv = (int)c.Nkv; p.D = (int)c.D;
  p.group = (int)(c.Hq / c.Hkv);
  p.causal = causal;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.n_chunks = (int)(c.D / kChunk);
  p.q_tiles = (int)((c.Nq + kTileRows - 1) / kTileRows);
  p.kv_tiles = (int)((c.Nkv + kTileRows - 1) / kTileRows);
  p.status = status;
  p.dropout = dropout;
  p.drop_t = drop_t; p.drop_seed_lo = seed_lo; p.drop_seed_hi = seed_hi; p.drop_off = drop_off;
  p.drop_scale = drop_scale;
  BwdMaps m;
  if ((rc = encode_map(&m.q, q)) || (rc = encode_map(&m.k, k)) || (rc = encode_map(&m.v, v)) ||
      (rc = encode_map(&m.dout, dout)) || (rc = encode_map(&m.q_half, q, kTileRows / 2)) ||
      (rc = encode_map(&m.k_half, k, kTileRows / 2)) || (rc = encode_map(&m.v_half, v, kTileRows / 2)) ||
      (rc = encode_map(&m.dout_half, dout, kTileRows / 2)))
    return rc;
  const size_t rows = (size_t)c.B * c.Hq * c.Nq;
  timing_begin();
  void* scratch = nullptr;
  if (scratch_alloc(&scratch, rows * 2 * sizeof(float), st) != cudaSuccess) return FFPA_ERR_CUDA;
  p.delta = static_cast<float*>(scratch);
  p.lse2 = p.delta + rows;
  cudaError_t e = launch_bwd(p, m, dtype_is_bf16(c.dtype), st);
  cudaError_t e2 = cudaFreeAsync(scratch, st);
  return cuda_rc(e != cudaSuccess ? e : e2);
}

}  // namespace

extern "C" int ffpa_fwd(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                        const ffpa_tensor_t* bias, int causal, float scale, const ffpa_tensor_t* out,
                        const ffpa_tensor_t* lse, ffpa_stream_t stream) {
  return fwd_impl(q, k, v, bias, causal, scale, nullptr, out, lse, stream);
}

extern "C" int ffpa_fwd_dropout(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                                const ffpa_tensor_t* bias, int causal, float scale, double dropout_p,
                                uint64_t seed, uint32_t offset, const ffpa_tensor_t* out, const ffpa_tensor_t* lse,
                                ffpa_stream_t stream) {
  const DropArgs d = {dropout_p, seed, offset};
  return fwd_impl(q, k, v, bias, causal, scale, &d, out, lse, stream);
}

extern "C" int ffpa_bwd(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                        const ffpa_tensor_t* bias, int causal, float scale, const ffpa_tensor_t* out,
                        const ffpa_tensor_t* lse, const ffpa_tensor_t* dout, const ffpa_tensor_t* dq,
                        const ffpa_tensor_t* dk, const ffpa_tensor_t* dv, ffpa_stream_t stream) {
  return bwd_impl(q, k, v, bias, causal, scale, nullptr, out, lse, dout, dq, dk, dv, stream);
}

extern "C" int ffpa_bwd_dropout(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                                const ffpa_tensor_t* bias, int causal, float scale, double dropout_p,
                                uint64_t seed, uint32_t offset, const ffpa_tensor_t* out, const ffpa_tensor_t* lse,
                                const ffpa_tensor_t* dout, const ffpa_tensor_t* dq, const ffpa_tensor_t* dk,
                                const ffpa_tensor_t* dv, ffpa_stream_t stream) {
  const DropArgs d = {dropout_p, seed, offset};
  return bwd_impl(q, k, v, bias, causal, scale, &d, out, lse, dout, dq, dk, dv, stream);
}

// Decode without allocation: validation and parameters as ffpa_fwd's decode
// path; the partials go to the library's fixed device array.
extern "C" int ffpa_fwd_decode_noalloc(const ffpa_tensor_t* q, const ffpa_tensor_t* k, const ffpa_tensor_t* v,
                                       const ffpa_tensor_t* bias, int causal, float scale,
                                       const ffpa_tensor_t* out, const ffpa_tensor_t* lse, ffpa_stream_t stream) {
  Common c;
  int rc = check_common(q, k, v, bias, scale, &c);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FFPA_ERR_INVALID_ARG;
  rc = check_bhnd(out, c.dtype, {c.B, c.Hq, c.Nq, c.D});
  if (rc) return rc;
  if (lse && (rc = check_lse(lse, c))) return rc;
  if (c.Nq > kDecodeMaxRows) return FFPA_ERR_UNSUPPORTED;
  int64_t bsb, bsh, bsq, bsk;
  bias_strides(bias, &bsb, &bsh, &bsq, &bsk);
  DecodeParams p = {};
  p.q = q->data;
  p.k = k->data;
  p.v = v->data;
  p.out = out->data;
  p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
  p.bias = bias ? static_cast<const float*>(bias->data) : nullptr;
  p.q_sb = q->stride[0]; p.q_sh = q->stride[1]; p.q_sn = q->stride[2];
  p.k_sb = k->stride[0]; p.k_sh = k->stride[1]; p.k_sn = k->stride[2];
  p.v_sb = v->stride[0]; p.v_sh = v->stride[1]; p.v_sn = v->stride[2];
  p.o_sb = out->stride[0]; p.o_sh = out->stride[1]; p.o_sn = out->stride[2];
  p.bias_sb = bsb; p.bias_sh = bsh; p.bias_sq = bsq; p.bias_sk = bsk;
  p.B = (int)c.B; p.Hq = (int)c.Hq; p.Hkv = (int)c.Hkv; p.Nq = (int)c.Nq; p.Nkv = (int)c.Nkv; p.D = (int)c.D;
  p.group = (int)(c.Hq / c.Hkv);
  p.causal = causal;
  p.scale_log2 = scale * kLog2e;
  p.heads_per_cta = decode_heads_per_cta(p.group, p.Nq, p.D);
  p.split_len = decode_split_len(c.B, c.Hq / p.heads_per_cta, c.Nkv);
  p.n_splits = (int)((c.Nkv + p.split_len - 1) / p.split_len);
  p.status = device_status_word();  // fetched with cudaGetSymbolAddress, no allocation
  if (!p.status) return FFPA_ERR_CUDA;
  if (decode_scratch_bytes(p) > decode_noalloc_capacity_bytes()) return FFPA_ERR_SCRATCH_LIMIT;
  timing_begin();
  return cuda_rc(launch_fwd_decode_noalloc(p, dtype_is_bf16(c.dtype), reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" const char* ffpa_status_string(int status) {
  switch (status) {
    case FFPA_OK: return "ok";
    case FFPA_ERR_INVALID_ARG: return "invalid argument";
    case FFPA_ERR_UNSUPPORTED: return "unsupported dtype, head dimension or layout";
    case FFPA_ERR_ALIGNMENT: return "pointer or stride not aligned for TMA (16 bytes)";
    case FFPA_ERR_CUDA: return "CUDA runtime or launch error";
    case FFPA_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case FFPA_ERR_SCRATCH_LIMIT: return "the call needs more than the fixed no-allocation scratch (8 MiB)";
    default: return "unknown status";
  }
}

extern "C" int ffpa_check_status(ffpa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FFPA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v)) != cudaSuccess) return FFPA_ERR_CUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)) != cudaSuccess) return FFPA_ERR_CUDA;
    return v == FFPA_DEV_TIMEOUT ? FFPA_ERR_TIMEOUT : FFPA_ERR_CUDA;
  }
  return FFPA_OK;
}

extern "C" int ffpa_set_timing_events(void* const* events, int count) {
  if (count < 0 || count > 8 || (count > 0 && !events)) return FFPA_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i)
    if (!events[i]) return FFPA_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) g_hook.ev[i] = static_cast<cudaEvent_t>(events[i]);
  g_hook.n = count;
  g_hook.next = 0;
  return FFPA_OK;
}

namespace ffpa {
namespace {
// One warp waits on an mbarrier that nothing arrives on; the bounded wait
// records FFPA_DEV_TIMEOUT and returns.
__global__ void selftest_wait_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status);
}
}  // namespace
}  // namespace ffpa

extern "C" int ffpa_selftest_wait_timeout(ffpa_stream_t stream) {
  uint32_t* status = device_status_word();
  if (!status) return FFPA_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? FFPA_OK : FFPA_ERR_CUDA;
}

extern "C" int ffpa_version(void) { return 100; }
