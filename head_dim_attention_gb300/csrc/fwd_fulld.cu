// Fused attention forward for D = 512: a CTA pair that holds ALL of O for
// one 128-row query tile.
//
// Same computation as fwd_main.cu and fwd_pair.cu (O = softmax(scale Q K^T +
// bias) V and the row logsumexp, online softmax over key tiles).  The other
// D = 512 flavour splits O's 512 columns between CTAs and so reduces S over
// the whole of D once per half; here a pair of CTAs issues tcgen05.mma
// cta_group::2 with M = 128, for which each SM receives 64 rows of the
// accumulator spread over all 128 TMEM lanes (lane r < 64: row r, the first
// N/2 columns; lane r + 64: row r, the other N/2).  A 128 x 512 fp32 O then
// takes 256 TMEM columns per SM, S is computed once per key tile, and the
// executed work is the algorithmic 4 Nq Nkv D per head plus the residual term
// of P where it is needed.
//
// Per CTA c of the pair (query rows q0 + 64c .. q0 + 64c + 63):
//   * Q resident in shared memory: 8 chunk tiles of 64 rows x 64 columns;
//   * key tiles of 128 keys: S = Q K^T with M=128, N=128: B split by N, this
//     CTA loads keys 64c .. 64c+63 of the tile (64 KB over all of D); TMEM S
//     buffer (64 columns): lane r holds keys 0..63 of row r, lane r + 64 keys
//     64..127 (double-buffered);
//   * softmax by 128 threads, two per row (thread t: row t mod 64, key half
//     t / 64); the row maximum is exchanged between the two through shared
//     memory, and each keeps its half's running sum, added at the end;
//   * P (and, on tiles that need it, its rounding residual) is written to
//     shared memory as the K-major A operand (64 rows x 128 keys, 16 KB): a
//     probe of the TMEM form of this MMA's A operand did not match the layout
//     S arrives in, so P goes through shared memory;
//   * O += P V: two MMAs per 16-key step (D columns 0..255 and 256..511),
//     M=128, N=256, B split by N: this CTA loads 128 of each half's columns
//     (128 keys x 256 columns = 64 KB per key tile); TMEM columns [0, 128)
//     hold D 128c'.. of half 0, [128, 256) of half 1 (c' = lane / 64).
// With Q (64 KB) and P (32 KB) resident, four 32 KB ring slots hold one key
// tile's K and V loads together.
//
// Warp roles: warps 0, 2, 3 TMA producers (each CTA its own halves), warp 1
// TMEM owner and, in the first CTA, the MMA issuer; warps 4-7 softmax.
// Synchronisation across the pair as in fwd_pair.cu: the first CTA's `full`
// barriers count both CTAs' bytes, its commits arrive on both CTAs' barriers,
// both CTAs' softmax warps arrive on its `p_ready`.  Every wait is bounded.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 256;
constexpr int kProducers = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kS0 = 256, kS1 = 320;      // S score buffers (64 columns each); O in [0, 256)
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLoFrac = 1.0f / 64.0f;       // residual term of P only where a weight exceeds this share
constexpr int kChunks = 8;                    // D = 512
constexpr int kKeys = 128;                    // keys per tile
constexpr int kHalfBytes = kChunkBytes / 2;   // 64 rows x 64 columns
constexpr int kQBytes = kChunks * kHalfBytes;  // 64 KB
constexpr int kPBytes = 2 * kHalfBytes;        // 64 rows x 128 keys, 16 KB
constexpr int kSlotBytes = 2 * kChunkBytes;    // 32 KB
constexpr int kStages = 4;
// shared memory: Q | P_hi | P_lo | ring | barriers + exchange
constexpr int kPHiOff = kQBytes, kPLoOff = kPHiOff + kPBytes, kRingOff = kPLoOff + kPBytes;
constexpr int kMiscOff = kRingOff + kStages * kSlotBytes;
constexpr int kSmemBytes = kMiscOff + 2048 + 1024;  // + alignment slack

struct Bars {
  int full, empty, q_full, s_full, p_ready, o_ready, mx, drain, count;
};
__host__ __device__ constexpr Bars bar_layout() {
  return Bars{0, kStages, 2 * kStages, 2 * kStages + 1, 2 * kStages + 3, 2 * kStages + 5, 2 * kStages + 6,
              2 * kStages + 8, 2 * kStages + 9};
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16)
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  else
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Row r of a K-major, 128-byte-swizzled tile of 64 rows x 64 16-bit values:
// its eight 16-byte granules sit at r*128 + ((g ^ (r & 7)) << 4).
__device__ __forceinline__ void store_row64(uint32_t tile, int r, const uint32_t (&w)[32]) {
  const uint32_t row = tile + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int g = 0; g < 8; ++g)
    st_shared_v4(row + ((static_cast<uint32_t>(g) ^ (r & 7)) << 4), w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_fulld_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                     const __grid_constant__ CUtensorMap map_v, const __grid_constant__ FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr Bars bl = bar_layout();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  volatile uint32_t* lo_flag = tmem_slot + 1;                         // [2], see fwd_pair.cu
  float* xm = reinterpret_cast<float*>(smem + kMiscOff + 512);         // [2][128] row-max exchange
  float* xl = xm + 256;                                                // [128] final row-sum exchange
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t base = smem_u32(smem);
  const uint32_t q_sm = base, phi_sm = base + kPHiOff, plo_sm = base + kPLoOff, ring_sm = base + kRingOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int qt = p.q_tiles - 1 - (static_cast<int>(blockIdx.x) >> 1);  // heavy causal tiles first
  const int q0 = qt * kTileRows;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / p.group;
  const int kv_end = p.causal ? min(p.Nkv, q0 + kTileRows) : p.Nkv;
  const int ntiles = (kv_end + kKeys - 1) / kKeys;
  uint32_t* status = p.status;
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(bl.full + i), 1);
      mbar_init(bar(bl.empty + i), 1);
    }
    mbar_init(bar(bl.q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.s_full + i), 1);
      mbar_init(bar(bl.p_ready + i), 8);  // four softmax warps in each CTA
      mbar_init(bar(bl.mx + i), 4);       // this CTA's four softmax warps
    }
    mbar_init(bar(bl.o_ready), 1);
    mbar_init(bar(bl.drain), 1);
    lo_flag[0] = 0;
    lo_flag[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    const int nprod = kProducers;  // <= kStages
    const int pi = (warp == 0) ? 0 : warp - 1;
    if (lane == 0) {
      tma_prefetch_desc(&map_qh);
      tma_prefetch_desc(&map_kh);
      tma_prefetch_desc(&map_v);
      if (pi == 0) {
        if (rank == 0) mbar_expect_tx(bar(bl.q_full), 2 * kQBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d_pair(q_sm + c * kHalfBytes, &map_qh, lead(bl.q_full), c * kChunk,
                           q0 + 64 * static_cast<int>(rank), h, b);
      }
      bool ok = true;
      uint32_t it = 0;
      // kind 0: K chunks 4m .. 4m+3 of this CTA's 64 keys of tile j (m = 0, 1);
      // kind 1: V chunks (this CTA's two of D half m) of the 128 keys of tile j
      auto slot = [&](int kind, int j, int m) {
        if (ok && static_cast<int>(it % nprod) == pi) {
          const uint32_t s = it % kStages, r = it / kStages;
          ok = mbar_wait(bar(bl.empty + s), (r & 1) ^ 1, status);
          if (ok) {
            if (rank == 0) mbar_expect_tx(bar(bl.full + s), 2 * kSlotBytes);
            const uint32_t dst = ring_sm + s * kSlotBytes, fb = lead(bl.full + s);
            if (kind == 0) {
              for (int i = 0; i < 4; ++i)
                tma_load_4d_pair(dst + i * kHalfBytes, &map_kh, fb, (4 * m + i) * kChunk,
                                 j * kKeys + 64 * static_cast<int>(rank), kvh, b);
            } else {
              for (int i = 0; i < 2; ++i)
                tma_load_4d_pair(dst + i * kChunkBytes, &map_v, fb, (4 * m + 2 * static_cast<int>(rank) + i) * kChunk,
                                 j * kKeys, kvh, b);
            }
          }
        }
        ++it;
      };
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles)
          for (int m = 0; m < 2; ++m) slot(0, j, m);
        if (j >= 1)
          for (int m = 0; m < 2; ++m) slot(1, j - 1, m);
      }
      for (uint32_t s = 0; s < static_cast<uint32_t>(kStages) && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / kStages) * kStages;
        if (static_cast<int>(last % nprod) == pi) mbar_wait(bar(bl.empty + s), (last / kStages) & 1, status);
      }
      if (pi == 0 && rank == 0) mbar_wait(bar(bl.q_full), 0, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (first CTA of the pair)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc_s = idesc_f16(BF16, 128, 128, false, false);   // 128 rows x 128 keys
      const uint32_t idesc_pv = idesc_f16(BF16, 128, 256, false, true);   // 128 rows x 256 O columns
      const uint64_t dq = sdesc_sw128(q_sm, 16, 1024);                     // Q chunks (64 rows), K-major
      const uint64_t dk = sdesc_sw128(ring_sm, 16, 1024);                  // K chunks (64 keys), K-major
      const uint64_t dv = sdesc_sw128(ring_sm, kChunkBytes, 1024);         // V chunks, MN-major
      const uint64_t dphi = sdesc_sw128(phi_sm, 16, 1024);                 // P (64 rows x 128 keys), K-major
      const uint64_t dplo = sdesc_sw128(plo_sm, 16, 1024);
      bool ok = mbar_wait(bar(bl.q_full), 0, status);
      tc_fence_after();
      uint32_t it = 0;
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles) {
          // S_j into buffer j & 1, which P_{j-2} no longer occupies (P lives in
          // shared memory; the softmax warps read S_{j-2} before P_{j-1} could
          // be issued).
          const uint32_t s_tm = tbase + ((j & 1) ? kS1 : kS0);
          for (int m = 0; m < 2 && ok; ++m) {
            const uint32_t s = it % kStages;
            ok = mbar_wait(bar(bl.full + s), (it / kStages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            for (int i = 0; i < 4; ++i) {
              const int c = 4 * m + i;
              const uint64_t a = sdesc_advance(dq, c * kHalfBytes);
              const uint64_t bd = sdesc_advance(dk, s * kSlotBytes + i * kHalfBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss_pair(s_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_s, (c | kk) != 0);
            }
            umma_commit_pair(bar(bl.empty + s), 3);
            ++it;
          }
          if (!ok) break;
          umma_commit_pair(bar(bl.s_full + (j & 1)), 3);
        }
        if (j >= 1) {
          const int t = j - 1;
          ok = mbar_wait(bar(bl.p_ready + (t & 1)), (t >> 1) & 1, status);
          if (!ok) break;
          tc_fence_after();
          const bool use_lo = lo_flag[t & 1] == static_cast<uint32_t>(t + 1);
          for (int dh = 0; dh < 2 && ok; ++dh) {
            const uint32_t s = it % kStages;
            ok = mbar_wait(bar(bl.full + s), (it / kStages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bd = sdesc_advance(dv, s * kSlotBytes);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // 16-key step within the tile
              const int k8 = kk;
              const uint32_t aoff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
              const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
              umma_ss_pair(tbase + 128 * dh, sdesc_advance(dphi, aoff), sdesc_advance(bd, k8 * 2048), idesc_pv, acc);
              if (use_lo)
                umma_ss_pair(tbase + 128 * dh, sdesc_advance(dplo, aoff), sdesc_advance(bd, k8 * 2048), idesc_pv, 1u);
            }
            umma_commit_pair(bar(bl.empty + s), 3);
            ++it;
          }
          if (!ok) break;
          umma_commit_pair(bar(bl.o_ready), 3);
        }
      }
      umma_commit_pair(bar(bl.drain), 1);
      mbar_wait(bar(bl.drain), 0, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / correction / epilogue
    const int t = tid - 128;      // TMEM lane
    const int r = t & 63;         // row within this CTA's 64
    const int kh = t >> 6;        // which 64 keys of each tile this thread scores
    const int row = q0 + 64 * static_cast<int>(rank) + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const float* bias_row = nullptr;
    if (p.bias)
      bias_row = p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(min(row, p.Nq - 1)) * p.bias_sq;
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t lo_flag_lead = rank == 0 ? 0u : mapa(smem_u32(const_cast<uint32_t*>(lo_flag)), 0);
    bool ok = true;
    float m_used = -INFINITY, l_sum = 0.f;  // l_sum: this thread's half of the row
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t s_col = (j & 1) ? kS1 : kS0;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.s_full + (j & 1)), (j >> 1) & 1, status));
      if (!ok) break;
      tc_fence_after();
      float s[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + s_col + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      const int kv0 = j * kKeys + 64 * kh;  // key of s[0]
      const bool masked = (kv0 + 64 > p.Nkv) || (p.causal && kv0 + 63 > row);
      const float c_scale = p.scale_log2;
      if (bias_row) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          s[i] = fmaf(__ldg(bias_row + static_cast<int64_t>(min(kv0 + i, p.Nkv - 1)) * p.bias_sk), kLog2e,
                      s[i] * c_scale);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] *= c_scale;
      }
      if (masked) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int kv = kv0 + i;
          if (kv >= p.Nkv || (p.causal && kv > row)) s[i] = -INFINITY;
        }
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
      const float m_half = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      // the row's maximum over both halves: exchange with the thread holding
      // the other 64 keys of this row (t ^ 64, in warp w ^ 2)
      xm[(j & 1) * 128 + t] = m_half;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bl.mx + (j & 1)));
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.mx + (j & 1)), (j >> 1) & 1, status));
      if (!ok) break;
      const float m_tile = fmaxf(m_half, xm[(j & 1) * 128 + (t ^ 64)]);
      float alpha = 1.f;
      bool rescale = false;
      if (m_used == -INFINITY) {
        m_used = m_tile;
      } else if (m_tile > m_used + kRescaleLog2) {
        alpha = ex2(m_used - m_tile);
        m_used = m_tile;
        rescale = true;
      }
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        s[i] = ex2(s[i] - m_ref);
        ls[i & 3] += s[i];
      }
      l_sum = l_sum * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      // residual term wanted where this half holds a weight above kLoFrac of
      // the half's running sum (a conservative stand-in for the row's sum)
      const bool warp_lo = __any_sync(0xffffffffu, ex2(m_half - m_ref) > kLoFrac * l_sum);
      if (j >= 1) {
        // P_j overwrites the shared-memory P that the P_{j-1} V product reads,
        // and the correction below rewrites O: wait for that product first.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.o_ready), (j - 1) & 1, status));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale) && j >= 1) {
        for (int c = 0; c < 8; ++c) {  // this lane's 256 O columns *= alpha
          uint32_t v[32];
          const uint32_t a = tbase + lane_off + c * 32;
          tmem_ld32(a, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(a, v);
        }
        tmem_st_wait();
      }
      // P of keys 64 kh .. 64 kh + 63 of row r: K-chunk kh of the P tile
      {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = s[2 * e], p1 = s[2 * e + 1];
          hi[e] = pack2<BF16>(p0, p1);
          if (warp_lo) {
            const float2 hv = unpack2<BF16>(hi[e]);
            lo[e] = pack2<BF16>(p0 - hv.x, p1 - hv.y);
          } else {
            lo[e] = 0u;
          }
        }
        store_row64(phi_sm + kh * kHalfBytes, r, hi);
        store_row64(plo_sm + kh * kHalfBytes, r, lo);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t pr_bar = lead(bl.p_ready + (j & 1));
        if (rank == 0) {
          if (warp_lo) lo_flag[j & 1] = static_cast<uint32_t>(j + 1);
          mbar_arrive(pr_bar);
        } else {
          if (warp_lo) st_cluster_u32(lo_flag_lead + 4 * (j & 1), static_cast<uint32_t>(j + 1));
          mbar_arrive_remote(pr_bar);
        }
      }
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      // the row's sum: this half's plus the partner's (same running max)
      xl[t] = l_sum;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bl.mx + (ntiles & 1)));
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.mx + (ntiles & 1)), (ntiles >> 1) & 1, status));
      const float l_row = l_sum + xl[t ^ 64];
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.o_ready), (ntiles - 1) & 1, status));
      if (ok) {
        tc_fence_after();
        const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
        typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
        T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + c * 32, v);
          tmem_ld_wait();
          if (row < p.Nq) {
            // TMEM column 32c + i of lane kh*64 + r is D column 256 (c / 4) + 128 kh + 32 (c % 4) + i
            const int d0 = 256 * (c >> 2) + 128 * kh + 32 * (c & 3);
            uint4* dst = reinterpret_cast<uint4*>(orow + d0);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 w;
              w.x = pack2<BF16>(__uint_as_float(v[8 * g + 0]) * inv_l, __uint_as_float(v[8 * g + 1]) * inv_l);
              w.y = pack2<BF16>(__uint_as_float(v[8 * g + 2]) * inv_l, __uint_as_float(v[8 * g + 3]) * inv_l);
              w.z = pack2<BF16>(__uint_as_float(v[8 * g + 4]) * inv_l, __uint_as_float(v[8 * g + 5]) * inv_l);
              w.w = pack2<BF16>(__uint_as_float(v[8 * g + 6]) * inv_l, __uint_as_float(v[8 * g + 7]) * inv_l);
              dst[g] = w;
            }
          }
        }
        if (kh == 0 && p.lse && row < p.Nq) {
          constexpr float kLn2 = 0.6931471805599453f;
          p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] =
              l_row > 0.f ? (m_used + __log2f(l_row)) * kLn2 : -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, kTmemCols);
  }
}

template <bool BF16>
cudaError_t launch_impl(const FwdParams& p_in, const FwdMaps& m, cudaStream_t st) {
  FwdParams p = p_in;
  p.stages = kStages;
  p.slot_chunks = 2;
  auto kern = fwd_fulld_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.q_tiles, p.Hq, p.B);  // (pair rank, query tile)
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  timing_mark(st);
  e = cudaLaunchKernelEx(&cfg, kern, m.q_half, m.k_half, m.v, p);
  timing_mark(st);
  return e;
}

}  // namespace

bool fwd_fulld_supported(const FwdParams& p) { return p.n_chunks == kChunks; }

cudaError_t launch_fwd_fulld(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_impl<true>(p, m, s) : launch_impl<false>(p, m, s);
}

}  // namespace ffpa
