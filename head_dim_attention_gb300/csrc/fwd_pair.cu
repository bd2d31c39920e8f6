// Fused attention forward, CTA-pair flavour, for D = 512.
//
// Same computation as fwd_main.cu (O = softmax(scale * Q K^T + bias) V and the
// row logsumexp, keys streamed in tiles of 128 with an online softmax), laid
// out for GB300's paired tensor cores.
//
// TMEM (512 fp32 columns per SM) cannot hold a 128 x 512 fp32 O accumulator
// next to the score tiles, so O is split by D in two halves of 256 columns
// (the FFPA pages' fine tiling along D, FFPA-Attn Performance Benchmarks page,
// "Why the Trends Look Like This"), and the scores are reduced over the whole
// of D by every CTA that owns a half.  In this flavour two CTAs that own the
// SAME half of D for two different 128-row query tiles form a cluster and
// issue their MMAs as one pair (tcgen05 cta_group::2, M = 256):
//   * S = Q K^T: each CTA supplies its own query tile (A, resident) and HALF
//     of the key tile (B, 64 keys x 512); each receives its 128 x 128 scores;
//   * O += P V: each CTA supplies its own P (A, from its TMEM) and HALF of the
//     V columns of the shared O half (B, 128 keys x 128); each accumulates its
//     128 x 256 slice of O.
// So every SM loads 96 KB per key tile instead of 192 KB, and its shared
// memory serves 3 KB of MMA operands per 64-row-equivalent step instead of 4.
//
// Two threads of the first CTA issue the pair's MMAs: a single thread spends
// longer issuing a pair MMA, and waiting on a barrier, than the tensor core
// needs for the MMA, so one issuer leaves the tensor core idle.  Thread A
// issues the S products from a ring of K tiles, thread B the P V products
// from a ring of V tiles; each ring has its own TMA producer.
//
// Warp roles (384 threads per CTA): warp 0 K producer, warp 3 V producer
// (each CTA loads its own halves), warp 1 TMEM owner (both CTAs) and, in the
// first CTA of the pair, MMA issuer A; warp 2 MMA issuer B (first CTA);
// warps 4-11 softmax / correction / epilogue for the CTA's own 128 query rows:
// warps 4-7 take keys 0..63 of every key tile and O columns 0..127 of the
// half, warps 8-11 keys 64..127 and O columns 128..255 (thread = row = TMEM
// lane; two warps per row quadrant, so each SM sub-partition runs two softmax
// warps that hide each other's latencies).  The two threads of a row swap
// their partial row maxima and sums through shared memory at a named barrier
// of the two warps.
//
// Synchronisation across the pair: the issuing CTA's `full` barriers count
// the bytes of both CTAs' loads; its commits arrive on the `empty`, `s_full`
// and `pv_done` barriers of both CTAs; both CTAs' softmax warps arrive on the
// issuing CTA's `p_ready`.  S_j and P_j share TMEM buffer j mod 2, so thread A
// writes S_j only after P_{j-2} V completed (pv_done of that buffer), and the
// softmax warps rescale O only after the previous P V completed.  Every wait
// is bounded (see ptx.cuh).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kS0 = 256, kS1 = 384;      // TMEM columns of the two S/P buffers; O in [0, 256)
constexpr float kRescaleLog2 = 8.0f;          // rescale O only when the max grows by > 2^8
constexpr float kLoFrac = 1.0f / 64.0f;       // see fwd_main.cu: residual term of P only where needed
constexpr int kChunks = 8;                    // D = 512: eight 64-column chunks
constexpr int kQBytes = kChunks * kChunkBytes;        // resident query tile, 128 KB
constexpr int kSlotBytes = 2 * kChunkBytes;           // ring slot: 4 half-key-tile K chunks or 2 V chunks
constexpr int kHalfChunkBytes = kChunkBytes / 2;      // 64 keys x 64 columns
constexpr int kKSlots = 2, kVSlots = 1;               // K ring (one key tile) and V ring

struct Bars {
  int full_k, empty_k, full_v, empty_v, q_full, s_full, p_ready, pv_done, drain_a, drain_b, count;
};
__host__ __device__ constexpr Bars bar_layout() {
  return Bars{0,
              kKSlots,
              2 * kKSlots,
              2 * kKSlots + kVSlots,
              2 * (kKSlots + kVSlots),
              2 * (kKSlots + kVSlots) + 1,  // 2
              2 * (kKSlots + kVSlots) + 3,  // 2
              2 * (kKSlots + kVSlots) + 5,  // 2
              2 * (kKSlots + kVSlots) + 7,
              2 * (kKSlots + kVSlots) + 8,
              2 * (kKSlots + kVSlots) + 9};
}

// Q, the rings, 256 bytes of barriers and flags, and the row-statistics
// exchange (2 x 2 x 128 floats).  There is no room for alignment padding: the
// kernel checks that dynamic shared memory starts on a 1024-byte boundary.
constexpr int kBarArea = 256, kXchBytes = 2 * 2 * 128 * 4;
__host__ __device__ constexpr int smem_bytes() {
  return kQBytes + (kKSlots + kVSlots) * kSlotBytes + kBarArea + kXchBytes;
}

// Named barrier of the two softmax warps of one row quadrant that returns the
// AND of their predicates (both warps then take the same branch).
__device__ __forceinline__ bool pair_bar_and(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
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

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kh,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the same in both CTAs of the pair: both leave here
    if (threadIdx.x == 0) record_error(p.status, FFPA_DEV_LAYOUT);
    return;
  }
  uint8_t* smem = smem_raw;
  constexpr Bars bl = bar_layout();
  static_assert(bl.count * 8 + 16 <= kBarArea, "barrier area");
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQBytes + (kKSlots + kVSlots) * kSlotBytes);
  float* xch = reinterpret_cast<float*>(smem + kQBytes + (kKSlots + kVSlots) * kSlotBytes + kBarArea);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  // lo_flag[t & 1] == t + 1: tile t carries the residual term of P.  Only the
  // issuing CTA's copy is read; the peer's softmax warps write it remotely.
  volatile uint32_t* lo_flag = tmem_slot + 1;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t q_sm = smem_u32(smem), ring_k = q_sm + kQBytes, ring_v = ring_k + kKSlots * kSlotBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const int cl = static_cast<int>(blockIdx.x) >> 1;
  const int dh = cl & 1;                    // which half of D (O columns) the pair owns
  const int npairs = (p.q_tiles + 1) >> 1;
  const int pr = npairs - 1 - (cl >> 1);    // query-tile pair, heavy causal pairs first
  const int q0 = (2 * pr + static_cast<int>(rank)) * kTileRows;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / p.group;
  // Both CTAs sweep the key tiles that the pair's later query tile needs.
  const int kv_end = p.causal ? min(p.Nkv, (2 * pr + 2) * kTileRows) : p.Nkv;
  const int ntiles = (kv_end + kTileRows - 1) / kTileRows;
  uint32_t* status = p.status;
  // A barrier of the issuing CTA, addressed from this CTA.
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  if (tid == 0) {
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(bar(bl.full_k + i), 1);
      mbar_init(bar(bl.empty_k + i), 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bar(bl.full_v + i), 1);
      mbar_init(bar(bl.empty_v + i), 1);
    }
    mbar_init(bar(bl.q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.s_full + i), 1);
      mbar_init(bar(bl.p_ready + i), 16);  // eight softmax warps in each CTA
      mbar_init(bar(bl.pv_done + i), 1);
    }
    mbar_init(bar(bl.drain_a), 1);
    mbar_init(bar(bl.drain_b), 1);
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

  if ((warp == 0 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ TMA producers (K: warp 0, V: warp 3)
    // This CTA's slot s is free once the pair's MMAs reading it completed (the
    // issuing CTA's commit arrives on empty[s] here); the bytes are counted on
    // the issuing CTA's full[s], which that CTA arms for both halves.
    const bool is_k = warp == 0;
    const int S = is_k ? kKSlots : kVSlots;
    const int full0 = is_k ? bl.full_k : bl.full_v, empty0 = is_k ? bl.empty_k : bl.empty_v;
    const uint32_t ring = is_k ? ring_k : ring_v;
    if (is_k) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_kh);
      if (rank == 0) mbar_expect_tx(bar(bl.q_full), 2 * kQBytes);
      for (int c = 0; c < kChunks; ++c)
        tma_load_4d_pair(q_sm + c * kChunkBytes, &map_q, lead(bl.q_full), c * kChunk, q0, h, b);
    } else {
      tma_prefetch_desc(&map_v);
    }
    bool ok = true;
    uint32_t it = 0;
    const int nslots = is_k ? 2 * ntiles : ntiles;
    for (int n = 0; n < nslots && ok; ++n) {
      const uint32_t s = it % S, r = it / S;
      ++it;
      ok = mbar_wait(bar(empty0 + s), (r & 1) ^ 1, status);
      if (!ok) break;
      if (rank == 0) mbar_expect_tx(bar(full0 + s), 2 * kSlotBytes);
      const uint32_t dst = ring + s * kSlotBytes, fb = lead(full0 + s);
      if (is_k) {
        // chunks 4m .. 4m+3 of this CTA's 64 keys of key tile n / 2 (m = n mod 2)
        const int m = n & 1, jt = n >> 1;
        for (int i = 0; i < 4; ++i)
          tma_load_4d_pair(dst + i * kHalfChunkBytes, &map_kh, fb, (4 * m + i) * kChunk,
                           jt * kTileRows + 64 * static_cast<int>(rank), kvh, b);
      } else {
        // this CTA's two V chunks of the pair's O half, key tile n
        for (int i = 0; i < 2; ++i)
          tma_load_4d_pair(dst + i * kChunkBytes, &map_v, fb, (4 * dh + 2 * static_cast<int>(rank) + i) * kChunk,
                           n * kTileRows, kvh, b);
      }
    }
    // Drain: wait for the last release of each slot, so no commit arrival is
    // in flight when the CTA exits.
    for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / S) * S;
      mbar_wait(bar(empty0 + s), (last / S) & 1, status);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer A: S_j = Q K_j^T
    constexpr uint32_t idesc_s = idesc_f16(BF16, 256, 128, false, false);  // 2 x 128 query rows x 128 keys
    const uint64_t dq = sdesc_sw128(q_sm, 16, 1024);                        // Q chunks, K-major
    const uint64_t dk = sdesc_sw128(ring_k, 16, 1024);                      // half-tile K chunks, K-major
    bool ok = mbar_wait(bar(bl.q_full), 0, status);
    tc_fence_after();
    uint32_t it = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      // S_j lands in the TMEM buffer that held P_{j-2}: wait for P_{j-2} V.
      if (j >= 2) {
        ok = mbar_wait(bar(bl.pv_done + (j & 1)), ((j - 2) >> 1) & 1, status);
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t s_tm = tbase + ((j & 1) ? kS1 : kS0);
      for (int m = 0; m < 2 && ok; ++m) {
        const uint32_t s = it % kKSlots;
        ok = mbar_wait(bar(bl.full_k + s), (it / kKSlots) & 1, status);
        ++it;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint64_t a = sdesc_advance(dq, (4 * m + i) * kChunkBytes);
          const uint64_t bd = sdesc_advance(dk, s * kSlotBytes + i * kHalfChunkBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_pair(s_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_s, (m | i | kk) != 0);
        }
        umma_commit_pair(bar(bl.empty_k + s), 3);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.s_full + (j & 1)), 3);
    }
    umma_commit_pair(bar(bl.drain_a), 1);
    mbar_wait(bar(bl.drain_a), 0, status);
  } else if (warp == 2 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer B: O += P_t V_t
    constexpr uint32_t idesc_pv = idesc_f16(BF16, 256, 256, false, true);  // 2 x 128 query rows x 256 O columns
    const uint64_t dv = sdesc_sw128(ring_v, kChunkBytes, 1024);            // V chunks, MN-major
    bool ok = true;
    uint32_t it = 0;
    for (int t = 0; t < ntiles && ok; ++t) {
      ok = mbar_wait(bar(bl.p_ready + (t & 1)), (t >> 1) & 1, status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t p_tm = tbase + ((t & 1) ? kS1 : kS0);
      const uint32_t s = it % kVSlots;
      ok = mbar_wait(bar(bl.full_v + s), (it / kVSlots) & 1, status);
      ++it;
      if (!ok) break;
      tc_fence_after();
      const uint64_t bd = sdesc_advance(dv, s * kSlotBytes);
      const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_ts_pair(tbase, p_tm + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv, acc0 | (kk > 0));
      if (lo_flag[t & 1] == static_cast<uint32_t>(t + 1)) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // the P_lo term
          umma_ts_pair(tbase, p_tm + 64 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv, 1u);
      }
      umma_commit_pair(bar(bl.empty_v + s), 3);
      umma_commit_pair(bar(bl.pv_done + (t & 1)), 3);
    }
    umma_commit_pair(bar(bl.drain_b), 1);
    mbar_wait(bar(bl.drain_b), 0, status);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / correction / epilogue
    const int wq = warp & 3;          // row quadrant (TMEM lanes 32 wq ..)
    const int kh = (warp - 4) >> 2;   // 0: keys 0..63 and O columns 0..127; 1: keys 64..127, O 128..255
    const int r = 32 * wq + lane;     // query row within this CTA's tile == TMEM lane
    const int row = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t nb = 1 + wq;       // named barrier of this quadrant's two warps
    float* xmax = xch + 0 * 256;      // [kh][row]
    float* xsum = xch + 1 * 256;
    const float* bias_row = nullptr;
    if (p.bias)
      bias_row = p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(min(row, p.Nq - 1)) * p.bias_sq;
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t p_ready_lead0 = lead(bl.p_ready), p_ready_lead1 = lead(bl.p_ready + 1);
    const uint32_t lo_flag_lead = rank == 0 ? 0u : mapa(smem_u32(const_cast<uint32_t*>(lo_flag)), 0);
    bool ok = true;
    float m_used = -INFINITY, l_own = 0.f, l_sum = 0.f;  // l_sum: both halves of the row
    for (int j = 0; j < ntiles; ++j) {
      const int t = j;
      const uint32_t s_col = (t & 1) ? kS1 : kS0;
      const bool got = __all_sync(0xffffffffu, mbar_wait(bar(bl.s_full + (t & 1)), (t >> 1) & 1, status));
      float s[64];
      if (got) {
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tbase + lane_off + s_col + 64 * kh, v0);
        tmem_ld32(tbase + lane_off + s_col + 64 * kh + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(v0[i]);
          s[32 + i] = __uint_as_float(v1[i]);
        }
      }
      const int kv0 = j * kTileRows + 64 * kh;  // this thread's first key of the tile
      const bool masked = (kv0 + 64 > p.Nkv) || (p.causal && kv0 + 63 > row);
      // Scores in the log2 domain: x = s scale log2e (+ bias log2e).  Without a
      // bias the scale is applied inside the exponent below (it is positive,
      // so the maximum of s gives the maximum of x).
      const float c_scale = bias_row ? 1.f : p.scale_log2;
      if (bias_row) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          s[i] = fmaf(__ldg(bias_row + static_cast<int64_t>(min(kv0 + i, p.Nkv - 1)) * p.bias_sk), kLog2e,
                      s[i] * p.scale_log2);
      }
      if (masked) {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int kv = kv0 + i;
          if (kv >= p.Nkv || (p.causal && kv > row)) s[i] = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
      xmax[128 * kh + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c_scale;
      ok = pair_bar_and(nb, got);  // both warps of the quadrant see the same outcome
      if (!ok) break;
      const float m_tile = fmaxf(xmax[r], xmax[128 + r]);
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
        s[i] = ex2(fmaf(s[i], c_scale, -m_ref));  // P, in place
        ls[i & 3] += s[i];
      }
      l_own = l_own * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      xsum[128 * kh + r] = l_own;
      pair_bar_and(nb, true);
      l_sum = xsum[r] + xsum[128 + r];
      // the residual term of P on this tile if some row's largest weight
      // exceeds 1/64 of its running sum (this tile included); the same in both
      // warps of a quadrant
      const bool warp_lo = __any_sync(0xffffffffu, ex2(m_tile - m_ref) > kLoFrac * l_sum);
      // The correction rewrites O: wait for P_{j-1} V first.  P_{j+1} V cannot
      // have completed yet, so the parity of that phase is unambiguous even
      // when earlier tiles skipped this wait.
      if (__any_sync(0xffffffffu, rescale) && j >= 1) {  // the same in both warps of the quadrant
        const bool done =
            __all_sync(0xffffffffu, mbar_wait(bar(bl.pv_done + ((t - 1) & 1)), ((t - 1) >> 1) & 1, status));
        ok = pair_bar_and(nb, done);
        if (!ok) break;
        tc_fence_after();
        for (int c = 0; c < 2; ++c) {  // this thread's 128 O columns *= alpha
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            const uint32_t a = tbase + lane_off + (2 * kh + c) * kChunk + hh * 32;
            tmem_ld32(a, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(a, v);
          }
        }
      }
      // P_j goes to the buffer S_j arrived in (its previous P V completed before
      // S_j was issued): the rounded value (columns 0..63) and, where needed, its
      // rounding residual (columns 64..127; zeros from warps that do not need
      // it); this thread's keys are columns 32 kh .. 32 kh + 31 of each.
      if (warp_lo) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = s[32 * g + 2 * e], p1 = s[32 * g + 2 * e + 1];
            hi[e] = pack2<BF16>(p0, p1);
            const float2 hv = unpack2<BF16>(hi[e]);
            lo[e] = pack2<BF16>(p0 - hv.x, p1 - hv.y);
          }
          tmem_st16(tbase + lane_off + s_col + 32 * kh + 16 * g, hi);
          tmem_st16(tbase + lane_off + s_col + 64 + 32 * kh + 16 * g, lo);
        }
      } else {
        uint32_t zero[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zero[e] = 0u;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t hi[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[e] = pack2<BF16>(s[32 * g + 2 * e], s[32 * g + 2 * e + 1]);
          tmem_st16(tbase + lane_off + s_col + 32 * kh + 16 * g, hi);
          tmem_st16(tbase + lane_off + s_col + 64 + 32 * kh + 16 * g, zero);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t pr_bar = (t & 1) ? p_ready_lead1 : p_ready_lead0;
        if (rank == 0) {
          if (warp_lo) lo_flag[t & 1] = static_cast<uint32_t>(t + 1);
          mbar_arrive(pr_bar);
        } else {
          if (warp_lo) st_cluster_u32(lo_flag_lead + 4 * (t & 1), static_cast<uint32_t>(t + 1));
          mbar_arrive_remote(pr_bar);  // release.cluster: the flag store is visible first
        }
      }
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      // the last P V of each buffer (their commits also arrive on the peer CTA)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.pv_done + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, status));
      if (ok && ntiles >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.pv_done + (ntiles & 1)), ((ntiles - 2) >> 1) & 1, status));
      if (ok) {
        tc_fence_after();
        const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
        typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
        T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
        for (int c = 2 * kh; c < 2 * kh + 2; ++c) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_off + c * kChunk + hh * 32, v);
            tmem_ld_wait();
            if (row < p.Nq) {
              uint4* dst = reinterpret_cast<uint4*>(orow + (4 * dh + c) * kChunk + hh * 32);
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
        }
        if (dh == 0 && kh == 0 && p.lse && row < p.Nq) {
          constexpr float kLn2 = 0.6931471805599453f;
          p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] =
              l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
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
  constexpr int smem = smem_bytes();
  static_assert(smem <= 232448, "227 KB opt-in per block");
  p.stages = kKSlots + kVSlots;
  p.slot_chunks = 2;
  auto kern = fwd_pair_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int npairs = (p.q_tiles + 1) / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * npairs, p.Hq, p.B);  // (pair rank, D half, query-tile pair)
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  timing_mark(st);
  e = cudaLaunchKernelEx(&cfg, kern, m.q, m.k_half, m.v, p);
  timing_mark(st);
  return e;
}

}  // namespace

bool fwd_pair_supported(const FwdParams& p) { return p.n_chunks == kChunks; }

cudaError_t launch_fwd_pair(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_impl<true>(p, m, s) : launch_impl<false>(p, m, s);
}

}  // namespace ffpa
