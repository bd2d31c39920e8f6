// Decode-shaped attention forward (few query rows, many keys) on sm_103a.
//
// With Nq <= 16 a tensor-core tile of 128 query rows would be mostly
// padding, and the work is bound by reading K and V from HBM once (the
// "decode-attn" case of the FFPA Attention Benchmark page, Nq/Nkv = 1/8192).
// So the keys are split into slices; each CTA takes one (batch, query head,
// slice), computes its scores with CUDA-core dot products, a local softmax and
// an unnormalised partial O, and a second kernel merges the slices with their
// (max, sum) statistics:
//     M = max_s m_s,  w_s = 2^(m_s - M),  O = sum_s w_s O_s / sum_s w_s l_s,
//     lse = (M + log2 sum_s w_s l_s) ln 2.
// The merge is exact (the same identity the online softmax uses).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kMaxRows = 16;  // Nq limit of this path
constexpr int kKeysPerIter = 4;

template <bool BF16>
struct Vec8 {
  // 8 consecutive elements (16 bytes) converted to fp32
  __device__ __forceinline__ static void load(const void* ptr, float (&f)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(ptr));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (BF16) {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
        const float2 x = __bfloat1622float2(h);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
      } else {
        const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
        const float2 x = __half22float2(h);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
      }
    }
  }
};

// One CTA per (split, query head, batch).  Shared memory: q rows as fp32
// [Nq][D] and the slice's scores [Nq][split_len].
template <bool BF16>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(16) float dsm[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / p.group;
  const int D = p.D, Nq = p.Nq, L = p.split_len;
  float* q_s = dsm;           // [Nq][D]
  float* sc = dsm + Nq * D;   // [Nq][L]
  float* stat = sc + Nq * L;  // [Nq][2]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kv_begin = split * L;
  const int kv_len = min(L, p.Nkv - kv_begin);
  typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;

  // q rows -> fp32 smem
  for (int i = tid; i < Nq * (D / 8); i += kDecThreads) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    float f[8];
    Vec8<BF16>::load(reinterpret_cast<const T*>(p.q) + b * p.q_sb + h * p.q_sh + static_cast<int64_t>(r) * p.q_sn + c,
                     f);
#pragma unroll
    for (int e = 0; e < 8; ++e) q_s[r * D + c + e] = f[e];
  }
  __syncthreads();

  // scores: warps stride over keys, lanes over D in 8-element groups
  const T* kbase = reinterpret_cast<const T*>(p.k) + b * p.k_sb + g * p.k_sh;
  const int groups = D / 8;  // 16-byte groups per row
  constexpr float kLog2e = 1.4426950408889634f;
  for (int j0 = warp * kKeysPerIter; j0 < kv_len; j0 += (kDecThreads / 32) * kKeysPerIter) {
    float acc[kKeysPerIter][kMaxRows];
#pragma unroll
    for (int u = 0; u < kKeysPerIter; ++u)
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) acc[u][r] = 0.f;
    for (int c = lane; c < groups; c += 32) {
      float kf[kKeysPerIter][8];
#pragma unroll
      for (int u = 0; u < kKeysPerIter; ++u) {
        const int j = min(j0 + u, kv_len - 1);
        Vec8<BF16>::load(kbase + static_cast<int64_t>(kv_begin + j) * p.k_sn + c * 8, kf[u]);
      }
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < Nq) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[r * D + c * 8]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[r * D + c * 8 + 4]);
#pragma unroll
          for (int u = 0; u < kKeysPerIter; ++u)
            acc[u][r] += qa.x * kf[u][0] + qa.y * kf[u][1] + qa.z * kf[u][2] + qa.w * kf[u][3] + qb.x * kf[u][4] +
                         qb.y * kf[u][5] + qb.z * kf[u][6] + qb.w * kf[u][7];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kKeysPerIter; ++u) {
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < Nq) {
          float v = acc[u][r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          const int j = j0 + u;
          if (lane == 0 && j < kv_len) {
            const int kv = kv_begin + j;
            float x = v * p.scale_log2;
            if (p.bias)
              x = fmaf(__ldg(p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(r) * p.bias_sq +
                             static_cast<int64_t>(kv) * p.bias_sk),
                       kLog2e, x);
            if (p.causal && kv > r) x = -INFINITY;
            sc[r * L + j] = x;
          }
        }
      }
    }
  }
  __syncthreads();

  // per-row max and sum over the slice (one warp per row)
  for (int r = warp; r < Nq; r += kDecThreads / 32) {
    float m = -INFINITY;
    for (int j = lane; j < kv_len; j += 32) m = fmaxf(m, sc[r * L + j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float mref = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
    for (int j = lane; j < kv_len; j += 32) {
      const float e = exp2f(sc[r * L + j] - mref);
      sc[r * L + j] = e;
      l += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) {
      stat[2 * r] = m;
      stat[2 * r + 1] = l;
    }
  }
  __syncthreads();

  // partial O: threads over D (8-element groups), loop over the slice's keys
  const T* vbase = reinterpret_cast<const T*>(p.v) + b * p.v_sb + g * p.v_sh;
  for (int c = tid; c < groups; c += kDecThreads) {
    float o[kMaxRows][8];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
    int j = 0;
    for (; j + 4 <= kv_len; j += 4) {
      float vf[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        Vec8<BF16>::load(vbase + static_cast<int64_t>(kv_begin + j + u) * p.v_sn + c * 8, vf[u]);
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < Nq) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float w = sc[r * L + j + u];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[r][e] = fmaf(w, vf[u][e], o[r][e]);
          }
        }
      }
    }
    for (; j < kv_len; ++j) {
      float vf[8];
      Vec8<BF16>::load(vbase + static_cast<int64_t>(kv_begin + j) * p.v_sn + c * 8, vf);
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r)
        if (r < Nq) {
          const float w = sc[r * L + j];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[r][e] = fmaf(w, vf[e], o[r][e]);
        }
    }
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < Nq) {
        float* dst = p.part_o + ((((static_cast<int64_t>(b) * p.Hq + h) * Nq + r) * p.n_splits + split) * D) + c * 8;
        reinterpret_cast<float4*>(dst)[0] = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(o[r][4], o[r][5], o[r][6], o[r][7]);
      }
    }
  }
  if (tid < Nq) {
    float* ml = p.part_ml + (((static_cast<int64_t>(b) * p.Hq + h) * Nq + tid) * p.n_splits + split) * 2;
    ml[0] = stat[2 * tid];
    ml[1] = stat[2 * tid + 1];
  }
}

// Streaming variant for Nq <= 2 (the decode case proper).  Each warp takes a
// contiguous eighth of the slice's keys and streams K and V rows together,
// U keys at a time (every lane holds G 16-byte groups of each row in flight),
// keeping an online softmax (running max m, sum l and unnormalised O) in
// registers; lane i owns elements 8(i + 32 k) .. +7 of D.  The eight warps
// then merge their (m, l, O) through shared memory into the slice's partial,
// which the combine kernel reads exactly as it reads the general kernel's.
template <int R, int G, int U, bool BF16>
__global__ void __launch_bounds__(kDecThreads) decode_stream_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(16) float wsm[];  // [8 warps][R][D] partial O, then [8][R] m and l
  const int split = blockIdx.x, b = blockIdx.z;
  // query heads h0 .. h0 + heads_per_cta - 1 share kv head g: row r of this
  // CTA is query row r % Nq of head h0 + r / Nq
  const int h0 = blockIdx.y * p.heads_per_cta, g = h0 / p.group;
  const int nrows = p.heads_per_cta * p.Nq;
  const int D = p.D, Nq = p.Nq, L = p.split_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = D / 8;
  const int kv_begin = split * L;
  const int kv_len = min(L, p.Nkv - kv_begin);
  const int per_warp = (L + 7) / 8;
  const int j_begin = warp * per_warp;
  const int j_end = min(kv_len, j_begin + per_warp);
  typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
  constexpr float kLog2e = 1.4426950408889634f;

  float qf[R][G][8];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int c = lane + 32 * k;
      if (r < nrows && c < groups)
        Vec8<BF16>::load(reinterpret_cast<const T*>(p.q) + b * p.q_sb + (h0 + r / Nq) * p.q_sh +
                             static_cast<int64_t>(r % Nq) * p.q_sn + c * 8,
                         qf[r][k]);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[r][k][e] = 0.f;
    }
  float m[R], l[R], o[R][G][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[r][k][e] = 0.f;
  }
  const T* kbase = reinterpret_cast<const T*>(p.k) + b * p.k_sb + g * p.k_sh;
  const T* vbase = reinterpret_cast<const T*>(p.v) + b * p.v_sb + g * p.v_sh;
  for (int j0 = j_begin; j0 < j_end; j0 += U) {
    // issue every load of the U keys (K and V rows) before using any of them
    uint4 kr[U][G], vr[U][G];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = kv_begin + min(j0 + u, j_end - 1);
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int c = min(lane + 32 * k, groups - 1);
        kr[u][k] = __ldg(reinterpret_cast<const uint4*>(kbase + row * p.k_sn + c * 8));
        vr[u][k] = __ldg(reinterpret_cast<const uint4*>(vbase + row * p.v_sn + c * 8));
      }
    }
    float s[U][R];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int r = 0; r < R; ++r) s[u][r] = 0.f;
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (lane + 32 * k < groups) {
          float kf[8];
          const uint32_t w[4] = {kr[u][k].x, kr[u][k].y, kr[u][k].z, kr[u][k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 x;
            if constexpr (BF16)
              x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            else
              x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            kf[2 * i] = x.x;
            kf[2 * i + 1] = x.y;
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) s[u][r] = fmaf(qf[r][k][e], kf[e], s[u][r]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s[u][r] += __shfl_xor_sync(0xffffffffu, s[u][r], off);
        const int kv = kv_begin + j0 + u;
        float x = s[u][r] * p.scale_log2;
        if (p.bias)
          x = fmaf(__ldg(p.bias + b * p.bias_sb + (h0 + r / Nq) * p.bias_sh + static_cast<int64_t>(r % Nq) * p.bias_sq +
                         static_cast<int64_t>(min(kv, p.Nkv - 1)) * p.bias_sk),
                   kLog2e, x);
        const bool valid = (j0 + u < j_end) && r < nrows && !(p.causal && kv > r % Nq);
        s[u][r] = valid ? x : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float mx = m[r];
#pragma unroll
      for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u][r]);
      if (mx == -INFINITY) continue;  // nothing visible yet for this row
      const float alpha = ex2(m[r] - mx);  // m[r] = -inf gives 0
      float pj[U];
      float ps = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        pj[u] = ex2(s[u][r] - mx);
        ps += pj[u];
      }
      l[r] = l[r] * alpha + ps;
      m[r] = mx;
#pragma unroll
      for (int k = 0; k < G; ++k) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[r][k][e] *= alpha;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const uint32_t w[4] = {vr[u][k].x, vr[u][k].y, vr[u][k].z, vr[u][k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float2 x;
            if constexpr (BF16)
              x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
            else
              x = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            o[r][k][2 * i] = fmaf(pj[u], x.x, o[r][k][2 * i]);
            o[r][k][2 * i + 1] = fmaf(pj[u], x.y, o[r][k][2 * i + 1]);
          }
        }
      }
    }
  }
  // merge the eight warps
  float* so = wsm;                  // [8][R][D]
  float* sm = wsm + 8 * R * D;      // [8][R]
  float* sl = sm + 8 * R;           // [8][R]
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int c = lane + 32 * k;
      if (c < groups) {
        float4* dst = reinterpret_cast<float4*>(so + (warp * R + r) * D + c * 8);
        dst[0] = make_float4(o[r][k][0], o[r][k][1], o[r][k][2], o[r][k][3]);
        dst[1] = make_float4(o[r][k][4], o[r][k][5], o[r][k][6], o[r][k][7]);
      }
    }
    if (lane == 0) {
      sm[warp * R + r] = m[r];
      sl[warp * R + r] = l[r];
    }
  }
  __syncthreads();
  for (int r = 0; r < nrows; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, sm[w * R + r]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    float wgt[8];
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      wgt[w] = ex2(sm[w * R + r] - Mref);  // -inf (empty warp) gives 0
      Ls += wgt[w] * sl[w * R + r];
    }
    float* dst = p.part_o + ((((static_cast<int64_t>(b) * p.Hq + h0 + r / Nq) * Nq + r % Nq) * p.n_splits + split) * D);
    for (int d = threadIdx.x * 4; d < D; d += kDecThreads * 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(so + (w * R + r) * D + d);
        acc.x = fmaf(wgt[w], v.x, acc.x);
        acc.y = fmaf(wgt[w], v.y, acc.y);
        acc.z = fmaf(wgt[w], v.z, acc.z);
        acc.w = fmaf(wgt[w], v.w, acc.w);
      }
      *reinterpret_cast<float4*>(dst + d) = acc;
    }
    if (threadIdx.x == 0) {
      float* ml = p.part_ml + (((static_cast<int64_t>(b) * p.Hq + h0 + r / Nq) * Nq + r % Nq) * p.n_splits + split) * 2;
      ml[0] = M;
      ml[1] = Ls;
    }
  }
}


// Streaming decode through shared memory (Nq <= 2, K and V rows contiguous).
// The register-fed kernel above keeps only 8 KB per warp in flight and walks
// its keys in dependent rounds, which left HBM at ~40% of its copy rate.  Here
// one thread streams the slice's K and V rows into a ring of shared-memory
// stages with 1-D bulk TMA copies (16 keys of K and of V per stage, three
// stages in flight per CTA), and the eight warps read them from shared memory:
// warp w scores keys 2w and 2w+1 of each stage and keeps its own online
// softmax, merged at the end exactly as above.
constexpr int kBulkStages = 3;
constexpr int kBulkKeys = 16;  // keys per stage

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

template <int R, int G, bool BF16>
__global__ void __launch_bounds__(kDecThreads) decode_bulk_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t bsm[];
  const int split = blockIdx.x, b = blockIdx.z;
  // query heads h0 .. h0 + heads_per_cta - 1 share kv head g: row r of this
  // CTA is query row r % Nq of head h0 + r / Nq
  const int h0 = blockIdx.y * p.heads_per_cta, g = h0 / p.group;
  const int nrows = p.heads_per_cta * p.Nq;
  const int D = p.D, Nq = p.Nq, L = p.split_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = D / 8;
  const int kv_begin = split * L;
  const int kv_len = min(L, p.Nkv - kv_begin);
  const int nst = (kv_len + kBulkKeys - 1) / kBulkKeys;
  const uint32_t half_bytes = static_cast<uint32_t>(kBulkKeys * D * 2);  // one stage's K (or V) rows
  const uint32_t stage_bytes = 2 * half_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bsm + kBulkStages * stage_bytes);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kBulkStages + s]); };
  const uint32_t ring = smem_u32(bsm);
  uint32_t* status = p.status;
  typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
  constexpr float kLog2e = 1.4426950408889634f;
  const T* kbase = reinterpret_cast<const T*>(p.k) + b * p.k_sb + g * p.k_sh + static_cast<int64_t>(kv_begin) * D;
  const T* vbase = reinterpret_cast<const T*>(p.v) + b * p.v_sb + g * p.v_sh + static_cast<int64_t>(kv_begin) * D;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBulkStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kDecThreads / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // stage i: keys 16 i .. 16 i + 15 of the slice (fewer in the last one)
  auto issue = [&](int i) {
    const int s = i % kBulkStages;
    const int n = min(kBulkKeys, kv_len - i * kBulkKeys);
    const uint32_t bytes = static_cast<uint32_t>(n * D * 2);
    mbar_expect_tx(full(s), 2 * bytes);
    bulk_load(ring + s * stage_bytes, kbase + static_cast<int64_t>(i) * kBulkKeys * D, bytes, full(s));
    bulk_load(ring + s * stage_bytes + half_bytes, vbase + static_cast<int64_t>(i) * kBulkKeys * D, bytes, full(s));
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(kBulkStages, nst); ++i) issue(i);

  float qf[R][G][8];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int c = lane + 32 * k;
      if (r < nrows && c < groups)
        Vec8<BF16>::load(reinterpret_cast<const T*>(p.q) + b * p.q_sb + (h0 + r / Nq) * p.q_sh +
                             static_cast<int64_t>(r % Nq) * p.q_sn + c * 8,
                         qf[r][k]);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[r][k][e] = 0.f;
    }
  float m[R], l[R], o[R][G][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[r][k][e] = 0.f;
  }
  bool ok = true;
  for (int i = 0; i < nst; ++i) {
    const int s = i % kBulkStages;
    ok = __all_sync(0xffffffffu, mbar_wait(full(s), (i / kBulkStages) & 1, status));
    if (!ok) break;
    const int n = min(kBulkKeys, kv_len - i * kBulkKeys);
    const uint8_t* kst = bsm + s * stage_bytes;
    const uint8_t* vst = kst + half_bytes;
    float sc[2][R];
    int jj[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int kk = 2 * warp + u;             // key within the stage
      jj[u] = min(kk, n - 1);                  // rows past the slice end read a valid row, weight 0
      const uint8_t* krow = kst + static_cast<size_t>(jj[u]) * D * 2;
#pragma unroll
      for (int r = 0; r < R; ++r) sc[u][r] = 0.f;
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int c = lane + 32 * k;
        if (c < groups) {
          const uint4 w4 = *reinterpret_cast<const uint4*>(krow + c * 16);
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
          float kf[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 x;
            if constexpr (BF16)
              x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            else
              x = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
            kf[2 * e] = x.x;
            kf[2 * e + 1] = x.y;
          }
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) sc[u][r] = fmaf(qf[r][k][e], kf[e], sc[u][r]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sc[u][r] += __shfl_xor_sync(0xffffffffu, sc[u][r], off);
        const int kv = kv_begin + i * kBulkKeys + kk;
        float x = sc[u][r] * p.scale_log2;
        if (p.bias)
          x = fmaf(__ldg(p.bias + b * p.bias_sb + (h0 + r / Nq) * p.bias_sh + static_cast<int64_t>(r % Nq) * p.bias_sq +
                         static_cast<int64_t>(min(kv, p.Nkv - 1)) * p.bias_sk),
                   kLog2e, x);
        const bool valid = kk < n && r < nrows && !(p.causal && kv > r % Nq);
        sc[u][r] = valid ? x : -INFINITY;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float mx = fmaxf(m[r], fmaxf(sc[0][r], sc[1][r]));
      if (mx == -INFINITY) continue;  // nothing visible yet for this row
      const float alpha = ex2(m[r] - mx);
      const float p0 = ex2(sc[0][r] - mx), p1 = ex2(sc[1][r] - mx);
      l[r] = l[r] * alpha + p0 + p1;
      m[r] = mx;
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int c = lane + 32 * k;
        if (c < groups) {
          const uint4 a4 = *reinterpret_cast<const uint4*>(vst + static_cast<size_t>(jj[0]) * D * 2 + c * 16);
          const uint4 b4 = *reinterpret_cast<const uint4*>(vst + static_cast<size_t>(jj[1]) * D * 2 + c * 16);
          const uint32_t wa[4] = {a4.x, a4.y, a4.z, a4.w}, wb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 xa, xb;
            if constexpr (BF16) {
              xa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
              xb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
            } else {
              xa = __half22float2(*reinterpret_cast<const __half2*>(&wa[e]));
              xb = __half22float2(*reinterpret_cast<const __half2*>(&wb[e]));
            }
            o[r][k][2 * e] = fmaf(p1, xb.x, fmaf(p0, xa.x, o[r][k][2 * e] * alpha));
            o[r][k][2 * e + 1] = fmaf(p1, xb.y, fmaf(p0, xa.y, o[r][k][2 * e + 1] * alpha));
          }
        }
      }
    }
    // release the stage; thread 0 refills it once all eight warps are done
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
    if (threadIdx.x == 0 && i + kBulkStages < nst) {
      ok = mbar_wait(empty(s), (i / kBulkStages) & 1, status);
      if (ok) issue(i + kBulkStages);
    }
  }
  // every issued stage was waited on above, so no copy is still in flight; the
  // ring's first bytes now take the warps' partials
  __syncthreads();
  float* so = reinterpret_cast<float*>(bsm);  // [8][R][D]
  float* sm = so + 8 * R * D;                 // [8][R]
  float* sl = sm + 8 * R;                     // [8][R]
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int c = lane + 32 * k;
      if (c < groups) {
        float4* dst = reinterpret_cast<float4*>(so + (warp * R + r) * D + c * 8);
        dst[0] = make_float4(o[r][k][0], o[r][k][1], o[r][k][2], o[r][k][3]);
        dst[1] = make_float4(o[r][k][4], o[r][k][5], o[r][k][6], o[r][k][7]);
      }
    }
    if (lane == 0) {
      sm[warp * R + r] = m[r];
      sl[warp * R + r] = l[r];
    }
  }
  __syncthreads();
  for (int r = 0; r < nrows; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, sm[w * R + r]);
    const float Mref = (M == -INFINITY) ? 0.f : M;
    float wgt[8];
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      wgt[w] = ex2(sm[w * R + r] - Mref);
      Ls += wgt[w] * sl[w * R + r];
    }
    float* dst = p.part_o + ((((static_cast<int64_t>(b) * p.Hq + h0 + r / Nq) * Nq + r % Nq) * p.n_splits + split) * D);
    for (int d = threadIdx.x * 4; d < D; d += kDecThreads * 4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(so + (w * R + r) * D + d);
        acc.x = fmaf(wgt[w], v.x, acc.x);
        acc.y = fmaf(wgt[w], v.y, acc.y);
        acc.z = fmaf(wgt[w], v.z, acc.z);
        acc.w = fmaf(wgt[w], v.w, acc.w);
      }
      *reinterpret_cast<float4*>(dst + d) = acc;
    }
    if (threadIdx.x == 0) {
      float* ml = p.part_ml + (((static_cast<int64_t>(b) * p.Hq + h0 + r / Nq) * Nq + r % Nq) * p.n_splits + split) * 2;
      ml[0] = M;
      ml[1] = Ls;
    }
  }
}

// Merge the slices.  One CTA per (row, 128-column chunk of D, query head,
// batch): the block reduces the slices' (m, l) to M and L, then warp w sums
// slices w, w+8, ... for its lane's four columns (all its loads in flight) and
// the eight warps' sums are added through shared memory.
constexpr int kCombThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red may still be read by a previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < kCombThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

template <bool BF16>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const __grid_constant__ DecodeParams p) {
  // Launched as a programmatic dependent of the split kernel: it may be
  // scheduled before that grid ends, and waits here until the split grid has
  // completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float red[kCombThreads / 32];
  __shared__ float4 part[kCombThreads / 32][32];
  const int S = p.n_splits, D = p.D;
  const int nd = (D + 127) / 128;
  const int chunk = blockIdx.x % nd, r = blockIdx.x / nd, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base = ((static_cast<int64_t>(b) * p.Hq + h) * p.Nq + r) * S;
  const float* ml = p.part_ml + base * 2;
  float m = -INFINITY;
  for (int s = threadIdx.x; s < S; s += kCombThreads) m = fmaxf(m, ml[2 * s]);
  const float M = block_reduce(m, true, red);
  const float Mref = (M == -INFINITY) ? 0.f : M;
  float ls = 0.f;
  for (int s = threadIdx.x; s < S; s += kCombThreads) ls += exp2f(ml[2 * s] - Mref) * ml[2 * s + 1];
  const float Lsum = block_reduce(ls, false, red);
  const int q4 = chunk * 32 + lane;  // this lane's float4 column
  const bool col = q4 * 4 < D;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col) {
#pragma unroll 4
    for (int s = warp; s < S; s += kCombThreads / 32) {
      const float w = exp2f(ml[2 * s] - Mref);
      const float4 o = *reinterpret_cast<const float4*>(p.part_o + (base + s) * D + q4 * 4);
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && col) {
    float4 t = part[0][lane];
#pragma unroll
    for (int w = 1; w < kCombThreads / 32; ++w) {
      t.x += part[w][lane].x;
      t.y += part[w][lane].y;
      t.z += part[w][lane].z;
      t.w += part[w][lane].w;
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(r) * p.o_sn + q4 * 4;
    if constexpr (BF16) {
      reinterpret_cast<__nv_bfloat162*>(orow)[0] = __floats2bfloat162_rn(t.x * inv, t.y * inv);
      reinterpret_cast<__nv_bfloat162*>(orow)[1] = __floats2bfloat162_rn(t.z * inv, t.w * inv);
    } else {
      reinterpret_cast<__half2*>(orow)[0] = __floats2half2_rn(t.x * inv, t.y * inv);
      reinterpret_cast<__half2*>(orow)[1] = __floats2half2_rn(t.z * inv, t.w * inv);
    }
  }
  if (chunk == 0 && threadIdx.x == 0 && p.lse) {
    constexpr float kLn2 = 0.6931471805599453f;
    p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + r] = Lsum > 0.f ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
  }
}

template <int R, int G, int U, bool BF16>
cudaError_t launch_stream(const DecodeParams& p, cudaStream_t st) {
  const size_t smem = (static_cast<size_t>(8) * R * p.D + 16 * R) * 4;
  auto k1 = decode_stream_kernel<R, G, U, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k1<<<dim3(p.n_splits, p.Hq / p.heads_per_cta, p.B), kDecThreads, smem, st>>>(p);
  return cudaSuccess;
}

template <int R, int G, bool BF16>
cudaError_t launch_bulk(const DecodeParams& p, cudaStream_t st) {
  const size_t ring = static_cast<size_t>(kBulkStages) * 2 * kBulkKeys * p.D * 2;
  const size_t merge = (static_cast<size_t>(8) * R * p.D + 16 * R) * 4;
  const size_t smem = (ring > merge ? ring : merge) + 2 * kBulkStages * 8;
  auto k1 = decode_bulk_kernel<R, G, BF16>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  k1<<<dim3(p.n_splits, p.Hq / p.heads_per_cta, p.B), kDecThreads, smem, st>>>(p);
  return cudaSuccess;
}

template <bool BF16>
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t st);

template <bool BF16>
cudaError_t launch_decode_impl(const DecodeParams& p, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  timing_mark(st);
  // rows of K and V contiguous (row stride D): the slice streams through
  // shared memory with bulk copies.  A CTA takes heads_per_cta query heads of
  // one kv head (decode_heads_per_cta), so its rows are their query rows.
  const bool rows_contiguous = p.k_sn == p.D && p.v_sn == p.D;
  const int nrows = p.heads_per_cta * p.Nq;
  if (nrows <= 4 && p.D <= 512 && rows_contiguous && p.split_len % kBulkKeys == 0) {
    e = nrows == 1   ? launch_bulk<1, 2, BF16>(p, st)
        : nrows == 2 ? launch_bulk<2, 2, BF16>(p, st)
                     : launch_bulk<4, 2, BF16>(p, st);
  } else if (nrows <= 4 && p.D <= 512) {
    e = nrows == 1   ? launch_stream<1, 2, 4, BF16>(p, st)
        : nrows == 2 ? launch_stream<2, 2, 4, BF16>(p, st)
                     : launch_stream<4, 2, 2, BF16>(p, st);
  } else if (nrows <= 2) {
    e = nrows == 1 ? launch_stream<1, 4, 2, BF16>(p, st) : launch_stream<2, 4, 2, BF16>(p, st);
  } else {
    if (p.heads_per_cta != 1) return cudaErrorInvalidValue;
    const size_t smem = (static_cast<size_t>(p.Nq) * p.D + static_cast<size_t>(p.Nq) * p.split_len + 2 * p.Nq) * 4;
    auto k1 = decode_split_kernel<BF16>;
    e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k1<<<dim3(p.n_splits, p.Hq, p.B), kDecThreads, smem, st>>>(p);
  }
  if (e != cudaSuccess) return e;
  timing_mark(st);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine<BF16>(p, st);
}

template <bool BF16>
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t st) {
  // programmatic dependent launch: the combine grid's launch overlaps the end
  // of the split grid (it waits for the split grid's results in the kernel)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Nq * ((p.D + 127) / 128), p.Hq, p.B);
  cfg.blockDim = dim3(kCombThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<BF16>, p);
  timing_mark(st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_decode(const DecodeParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_decode_impl<true>(p, s) : launch_decode_impl<false>(p, s);
}

cudaError_t launch_decode_combine(const DecodeParams& p, bool bf16, cudaStream_t s) {
  return bf16 ? launch_combine<true>(p, s) : launch_combine<false>(p, s);
}

// Query heads one decode CTA takes: the whole GQA group when its rows (group
// x Nq) fit the register-fed kernels (K and V are then read once per group
// instead of once per query head), else one.
int decode_heads_per_cta(int group, int Nq, int D) {
  const int rows = group * Nq;
  return (rows <= 4 && D <= 512) || rows <= 2 ? group : 1;
}

}  // namespace ffpa

// ---------------------------------------------------------------------------
// Decode without allocation (ffpa_fwd_decode_noalloc).
//
// Some callers cannot allocate device memory while they run attention: code
// that runs inside another framework's memory pool, or a serving loop that
// must not call into the CUDA allocator on its hot path.  For them the decode
// partials live in this fixed, file-scope device array instead of
// cudaMallocAsync memory.  Every GPU that loads the library holds the array
// until the process exits.  All calls share it: the split kernel overwrites
// every partial the merge kernel reads, so nothing has to start at zero, and
// two such calls whose work overlaps on the GPU (other streams, other host
// threads) race on the array.
#include <mutex>

namespace ffpa {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

size_t decode_noalloc_capacity_bytes() { return kNoAllocScratchBytes; }

// Bytes of partials a decode call needs: (D + 2) floats per (b, h, row, slice).
size_t decode_scratch_bytes(const DecodeParams& p) {
  const size_t rows = static_cast<size_t>(p.B) * p.Hq * p.Nq * p.n_splits;
  return rows * (static_cast<size_t>(p.D) + 2) * sizeof(float);
}

// The array's device address on the current device.  In host code the name
// g_noalloc_scratch is only a host-side stand-in, so the address is fetched
// with cudaGetSymbolAddress once per device (on that device's first call) and
// cached.
static cudaError_t noalloc_scratch_address(float** out) {
  static std::mutex mu;
  static float* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    cache[dev] = static_cast<float*>(ptr);
  }
  *out = cache[dev];
  return cudaSuccess;
}

cudaError_t launch_fwd_decode_noalloc(const DecodeParams& p_in, bool bf16, cudaStream_t s) {
  if (decode_scratch_bytes(p_in) > kNoAllocScratchBytes) return cudaErrorInvalidValue;
  float* base = nullptr;
  cudaError_t e = noalloc_scratch_address(&base);
  if (e != cudaSuccess) return e;
  DecodeParams p = p_in;
  const size_t rows = static_cast<size_t>(p.B) * p.Hq * p.Nq * p.n_splits;
  p.part_o = base;
  p.part_ml = base + rows * p.D;  // D is a multiple of 64: 256-byte aligned
  return launch_fwd_decode(p, bf16, s);
}

}  // namespace ffpa
