// Fused attention forward for D = 704..1024 on clusters of four CTAs (two CTA
// pairs) per 128-row query tile, in which one pair computes the scores and the
// other accumulates O.
//
// Same computation as fwd_fulld.cu: O = softmax(scale Q K^T + bias) V and the
// row logsumexp, keys in tiles of 128 with an online softmax.  Above D = 512 a
// pair cannot hold Q, the score tiles and all of O (128 x D fp32 takes D / 2
// TMEM columns per SM in the M = 128 pair layout), and splitting O's columns
// between pairs makes every pair recompute S over all of D.  Here the work of a
// key tile is split by product instead (FFPA Attention Benchmark page, "More
// Benchmark": the SM100 2-CTA path, carried above D = 512):
//   pair A (cluster ranks 0, 1): Q resident (up to 12 of its 64-column chunks
//          in TMEM as the TS-form operand, the rest in shared memory);
//          S_j = Q K_j^T, the online softmax, P_j (and, where needed, the
//          rounding residual of P_j) -> pair B, with each row's rescale factor
//          and running sum;
//   pair B (ranks 2, 3): all of O in TMEM (D / 2 columns per SM, in blocks of
//          up to 256 O columns per MMA); before P_j V_j it applies pair A's
//          rescale factor to O's rows (only when a row's maximum grew by more
//          than 2^8), then O += P_j V_j (+ P_lo V_j); the epilogue divides by
//          the last running sum.
// S and P V are each computed once: 4 Nq Nkv D per head (plus the residual
// term on part of the tiles), against 6 for two O-split pairs at D = 1024.
//
// Layout within a pair (tcgen05 cta_group::2, M = 128): CTA c (c = rank & 1)
// holds query rows q0 + 64c .. q0 + 64c + 63 across all 128 TMEM lanes.  CTA r
// of pair A and CTA r + 2 of pair B hold the same rows; each tile's message
// goes between those two: every softmax warp of pair A writes its 32 rows x 64
// keys of P_hi and P_lo (4 KB each, K-major, 128-byte swizzle, the layout pair
// B's MMAs read as the A operand), its rows' (alpha, l) and its residual flag
// into a local staging buffer and copies them with bulk copies into the other
// CTA, whose barrier counts the bytes (33,344 per CTA and tile).
//
// Signals across the pairs: rfull[b] (bytes, armed by a thread of the
// receiving CTA); ready[b] (pair B's warps of both CTAs have read the factors
// and rescaled O; the second CTA's relay forwards, with its residual flag);
// rfree[b] (pair B's P V commit, multicast to pair A: buffer b may be refilled).
//
// Warps: 0 K producer and Q loader (pair A), 1 TMEM owner + MMA issuer (first
// CTA of a pair), 2 relay (second CTA of pair B), 3 V producer (pair B), 4-7
// softmax (pair A) or rescale and epilogue (pair B).  Every wait is bounded
// (ptx.cuh).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;          // rescale O only when the max grows by > 2^8
constexpr float kLoFrac = 1.0f / 64.0f;       // residual term of P only where a weight exceeds this share
constexpr int kHalfBytes = kChunkBytes / 2;   // 64 rows x 64 columns, 8 KB
constexpr int kPBytes = 2 * kHalfBytes;       // 64 rows x 128 keys, 16 KB
constexpr int kSlice = kHalfBytes / 2;        // one warp's 32 rows x 64 keys, 4 KB
constexpr int kStatOff = 2 * kPBytes;         // message: P_hi | P_lo | (alpha, l) x 64 rows | 4 flag granules
constexpr int kFlagOff = kStatOff + 64 * 8;
constexpr int kMsgBytes = kFlagOff + 4 * 16;  // 33,344
constexpr int kMsgStride = 33 * 1024;
constexpr int kNbuf = 2;                      // staging buffers (pair A) and receive buffers (pair B)
constexpr int kSlotBytes = 2 * kChunkBytes;   // 32 KB ring slots

template <int NC>
struct Shape {
  static_assert(NC >= 11 && NC <= 16, "D = 704 .. 1024");
  static constexpr int kD = 64 * NC;
  static constexpr uint32_t kS0 = 0, kS1 = 64, kQt = 128;      // pair A's TMEM: scores, then Q
  static constexpr int kQtc = NC < 12 ? NC : 12;               // Q chunks in TMEM
  static constexpr int kQBytes = (NC - kQtc) * kHalfBytes;     // the rest in shared memory
  static constexpr int kKSlotsPerTile = (NC + 3) / 4;          // pair A: four 8 KB K chunks per slot
  static constexpr int kNblk = (kD + 255) / 256;               // pair B: O blocks of up to 256 columns
  static constexpr int kSlots = NC == 16 ? 3 : 4;              // pair A's K ring
  static constexpr int kSlotsB = 4;                            // pair B's V ring
  // shared memory, pair A: Q rest | staging buffers | K ring; pair B: receive
  // buffers | V ring (over pair A's Q region too); then barriers and the row exchange
  static constexpr int kBufOff = kQBytes;
  static constexpr int kRingOff = kBufOff + kNbuf * kMsgStride;
  static constexpr int kRingOffB = kNbuf * kMsgStride;
  static constexpr int kMiscOff = kRingOff + kSlots * kSlotBytes > kRingOffB + kSlotsB * kSlotBytes
                                      ? kRingOff + kSlots * kSlotBytes
                                      : kRingOffB + kSlotsB * kSlotBytes;
  static constexpr int kSmemBytes = kMiscOff + 512 + 2 * 128 * 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "227 KB per CTA");
  static_assert(kQt + 32 * kQtc <= kTmemCols, "pair A's TMEM");
};

struct Bars {
  int full_r, empty_r, q_full, s_full, s_free, rfull, ready, ready_local, rfree, pv_done, drain, count;
};
// rings: up to four slots; s_*: one per score buffer; the rest one per message buffer
__host__ __device__ constexpr Bars bar_layout() { return Bars{0, 4, 8, 9, 11, 13, 15, 17, 19, 21, 23, 24}; }
static_assert(bar_layout().count * 8 + 16 <= 512, "barrier area");

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
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_v2f(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ float2 ld_shared_v2f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Row r of a K-major, 128-byte-swizzled tile of 64 rows x 64 16-bit values.
__device__ __forceinline__ void store_row64(uint32_t tile, int r, const uint32_t (&w)[32]) {
  const uint32_t row = tile + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int g = 0; g < 8; ++g)
    st_shared_v4(row + ((static_cast<uint32_t>(g) ^ static_cast<uint32_t>(r & 7)) << 4), w[4 * g], w[4 * g + 1],
                 w[4 * g + 2], w[4 * g + 3]);
}

// Named barrier of the two softmax warps that hold the two key halves of the
// same rows; returns the AND of their predicates.
__device__ __forceinline__ bool pair_bar_and(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

template <int NC, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_xch_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ FwdParams p) {
  using G = Shape<NC>;
  constexpr int kQtc = G::kQtc, kSlots = G::kSlots, kSlotsB = G::kSlotsB, kNblk = G::kNblk;
  constexpr Bars bl = bar_layout();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  // lo_peer[b] == j + 1: the second CTA of pair B received a residual term with tile j
  volatile uint32_t* lo_peer = tmem_slot + 1;
  float* xmax = reinterpret_cast<float*>(smem + G::kMiscOff + 512);  // [128]: by TMEM lane
  float* xsum = xmax + 128;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t base = smem_u32(smem);
  const uint32_t q_sm = base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0, 1: pair A (scores); 2, 3: pair B (O)
  const bool is_b = rank >= 2;
  const uint32_t pr = rank & 1, lead_rank = rank & 2, other = rank ^ 2;
  // message buffers (staging in pair A, receive in pair B) and the ring
  const uint32_t buf_sm = base + (is_b ? 0 : G::kBufOff);
  const uint32_t ring = base + (is_b ? G::kRingOffB : G::kRingOff);
  const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);
  const uint16_t other_mask = static_cast<uint16_t>(3u << (lead_rank ^ 2));
  const int qt = p.q_tiles - 1 - static_cast<int>(blockIdx.x >> 2);  // heavy causal tiles first
  const int q0 = qt * kTileRows;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / p.group;
  const int kv_end = p.causal ? min(p.Nkv, q0 + kTileRows) : p.Nkv;
  const int ntiles = (kv_end + kTileRows - 1) / kTileRows;
  uint32_t* status = p.status;
  auto lead = [&](int i) { return pr == 0 ? bar(i) : mapa(bar(i), lead_rank); };

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(bl.full_r + i), 1);
      mbar_init(bar(bl.empty_r + i), 1);
    }
    // Q ready (pair A): the armed TMA bytes of Q's shared-memory chunks and the
    // eight softmax warps of the pair that wrote the TMEM chunks
    mbar_init(bar(bl.q_full), 1 + 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.s_full + i), 1);
      mbar_init(bar(bl.s_free + i), 8);       // four softmax warps in each CTA of pair A
      mbar_init(bar(bl.rfull + i), 1);        // (pair B) the message's bytes
      mbar_init(bar(bl.ready + i), 5);        // (pair B) four local warps + the second CTA's relay
      mbar_init(bar(bl.ready_local + i), 4);  // (pair B, second CTA) its four warps
      mbar_init(bar(bl.rfree + i), 1);        // (pair A) pair B's P V commit
      mbar_init(bar(bl.pv_done + i), 1);      // (pair B) this pair's P V commit
      lo_peer[i] = 0;
    }
    mbar_init(bar(bl.drain), 1);
    // the first use of each receive buffer: this CTA expects one message
    if (is_b)
      for (int i = 0; i < kNbuf; ++i) mbar_expect_tx(bar(bl.rfull + i), kMsgBytes);
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

  if (!is_b && warp == 0 && lane == 0) {
    // ------------------------------------------------------------ pair A: Q (shared-memory chunks) and the K ring
    // This CTA's slot s is free once the pair's MMAs reading it completed (the
    // first CTA's commit arrives here); the bytes of both CTAs are counted on
    // the first CTA's full[s].
    tma_prefetch_desc(&map_qh);
    tma_prefetch_desc(&map_kh);
    if (pr == 0) mbar_expect_tx(bar(bl.q_full), 2 * G::kQBytes);
    for (int c = kQtc; c < NC; ++c)
      tma_load_4d_pair(q_sm + (c - kQtc) * kHalfBytes, &map_qh, lead(bl.q_full), c * kChunk,
                       q0 + 64 * static_cast<int>(pr), h, b);
    bool ok = true;
    uint32_t it = 0;
    for (int n = 0; n < G::kKSlotsPerTile * ntiles && ok; ++n) {
      const uint32_t s = it % kSlots, rr = it / kSlots;
      ++it;
      ok = mbar_wait<false>(bar(bl.empty_r + s), (rr & 1) ^ 1, status);
      if (!ok) break;
      const int j = n / G::kKSlotsPerTile, m = n % G::kKSlotsPerTile;
      const int nk = min(4, NC - 4 * m);  // K chunks 4m .. 4m + nk - 1 of this CTA's 64 keys of key tile j
      if (pr == 0) mbar_expect_tx(bar(bl.full_r + s), 2 * nk * kHalfBytes);
      const uint32_t dst = ring + s * kSlotBytes, fb = lead(bl.full_r + s);
      for (int i = 0; i < nk; ++i)
        tma_load_4d_pair(dst + i * kHalfBytes, &map_kh, fb, (4 * m + i) * kChunk,
                         j * kTileRows + 64 * static_cast<int>(pr), kvh, b);
    }
    for (uint32_t s = 0; s < static_cast<uint32_t>(kSlots) && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / kSlots) * kSlots;
      mbar_wait<false>(bar(bl.empty_r + s), (last / kSlots) & 1, status);
    }
  } else if (is_b && warp == 3 && lane == 0) {
    // ------------------------------------------------------------ pair B: the V ring
    // one slot per O block and key tile: this CTA's half of the block's
    // columns (one or two 64-column chunks) over the tile's 128 keys
    tma_prefetch_desc(&map_v);
    bool ok = true;
    uint32_t it = 0;
    for (int n = 0; n < kNblk * ntiles && ok; ++n) {
      const uint32_t s = it % kSlotsB, rr = it / kSlotsB;
      ++it;
      ok = mbar_wait<false>(bar(bl.empty_r + s), (rr & 1) ^ 1, status);
      if (!ok) break;
      const int j = n / kNblk, nb = n % kNblk;
      const int w = min(256, G::kD - 256 * nb);
      const int nv = w > 128 ? 2 : 1;  // chunks per CTA: the block's N = 128 nv columns, split over the pair
      if (pr == 0) mbar_expect_tx(bar(bl.full_r + s), 2 * nv * kChunkBytes);
      const uint32_t dst = ring + s * kSlotBytes, fb = lead(bl.full_r + s);
      for (int i = 0; i < nv; ++i)
        tma_load_4d_pair(dst + i * kChunkBytes, &map_v, fb, 256 * nb + (nv * static_cast<int>(pr) + i) * kChunk,
                         j * kTileRows, kvh, b);
    }
    for (uint32_t s = 0; s < static_cast<uint32_t>(kSlotsB) && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / kSlotsB) * kSlotsB;
      mbar_wait<false>(bar(bl.empty_r + s), (last / kSlotsB) & 1, status);
    }
  } else if (!is_b && warp == 1 && lane == 0 && pr == 0) {
    // ------------------------------------------------------------ pair A's MMA issuer: S_j = Q K_j^T
    constexpr uint32_t idesc_s = idesc_f16(BF16, 128, 128, false, false);  // 128 rows x 128 keys
    const uint64_t dq = sdesc_sw128(q_sm, 16, 1024);                        // Q chunks (64 rows), K-major
    const uint64_t dk = sdesc_sw128(ring, 16, 1024);                        // K chunks (64 keys), K-major
    bool ok = mbar_wait<false>(bar(bl.q_full), 0, status);
    tc_fence_after();
    uint32_t it = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      if (j >= 2) {
        // S_j goes to the buffer S_{j-2} used: the softmax warps have copied it out
        ok = mbar_wait<false>(bar(bl.s_free + (j & 1)), ((j - 2) >> 1) & 1, status);
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t s_tm = tbase + ((j & 1) ? G::kS1 : G::kS0);
#pragma unroll
      for (int m = 0; m < G::kKSlotsPerTile; ++m) {
        const uint32_t s = it % kSlots;
        ok = mbar_wait<false>(bar(bl.full_r + s), (it / kSlots) & 1, status);
        ++it;
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int x = 4 * m + i;  // chunk of D
          if (x >= NC) break;
          const uint64_t bd = sdesc_advance(dk, s * kSlotBytes + i * kHalfBytes);
          if (x < kQtc) {  // Q from TMEM (8 columns per 16-column step)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ts_pair(s_tm, tbase + G::kQt + 32 * x + 8 * kk, sdesc_advance(bd, kk * 32), idesc_s,
                           (x | kk) != 0);
          } else {  // Q from shared memory
            const uint64_t a = sdesc_advance(dq, (x - kQtc) * kHalfBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_pair(s_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_s, 1u);
          }
        }
        umma_commit_pair(bar(bl.empty_r + s), pair_mask);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.s_full + (j & 1)), pair_mask);
    }
    umma_commit_pair(bar(bl.drain), static_cast<uint16_t>(1u << rank));
    mbar_wait<false>(bar(bl.drain), 0, status);
  } else if (is_b && warp == 1 && lane == 0 && pr == 0) {
    // ------------------------------------------------------------ pair B's MMA issuer: O += P_j V_j (+ P_lo V_j)
    constexpr uint32_t idesc_256 = idesc_f16(BF16, 128, 256, false, true);  // 128 rows x 256 O columns
    constexpr uint32_t idesc_128 = idesc_f16(BF16, 128, 128, false, true);
    const uint64_t dv = sdesc_sw128(ring, kChunkBytes, 1024);  // V chunk pairs, MN-major
    const uint64_t dp = sdesc_sw128(buf_sm, 16, 1024);         // received P (64 rows x 128 keys), K-major
    bool ok = true;
    uint32_t it = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int rb = j % kNbuf;
      // both CTAs' warps have read the message and rescaled O where it asked
      ok = mbar_wait<false>(bar(bl.ready + rb), (j / kNbuf) & 1, status);
      if (!ok) break;
      tc_fence_after();
      // the residual term: this CTA's message flags or the second CTA's (forwarded)
      const uint32_t fl = buf_sm + rb * kMsgStride + kFlagOff;
      const bool use_lo = (ld_shared_u32(fl) | ld_shared_u32(fl + 16) | ld_shared_u32(fl + 32) |
                           ld_shared_u32(fl + 48)) != 0 ||
                          lo_peer[rb] == static_cast<uint32_t>(j + 1);
      const uint64_t dphi = sdesc_advance(dp, rb * kMsgStride), dplo = sdesc_advance(dphi, kPBytes);
      for (int nb = 0; nb < kNblk && ok; ++nb) {
        const uint32_t s = it % kSlotsB;
        ok = mbar_wait<false>(bar(bl.full_r + s), (it / kSlotsB) & 1, status);
        ++it;
        if (!ok) break;
        tc_fence_after();
        const uint64_t bd = sdesc_advance(dv, s * kSlotBytes);
        const uint32_t o_tm = tbase + 128 * nb;
        const uint32_t idesc = min(256, G::kD - 256 * nb) > 128 ? idesc_256 : idesc_128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // 16-key steps: P subtile ks / 4, V rows 16 ks ..
          umma_ss_pair(o_tm, sdesc_advance(dphi, (ks >> 2) * kHalfBytes + (ks & 3) * 32),
                       sdesc_advance(bd, ks * 2048), idesc, (j > 0 || ks > 0) ? 1u : 0u);
        if (use_lo) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_ss_pair(o_tm, sdesc_advance(dplo, (ks >> 2) * kHalfBytes + (ks & 3) * 32),
                         sdesc_advance(bd, ks * 2048), idesc, 1u);
        }
        umma_commit_pair(bar(bl.empty_r + s), pair_mask);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.pv_done + rb), pair_mask);  // O holds P_j V_j
      umma_commit_pair(bar(bl.rfree + rb), other_mask);   // pair A may refill buffer rb
    }
    umma_commit_pair(bar(bl.drain), static_cast<uint16_t>(1u << rank));
    mbar_wait<false>(bar(bl.drain), 0, status);
  } else if (is_b && warp == 2 && lane == 0 && pr == 1) {
    // ------------------------------------------------------------ pair B's relay for its first CTA
    const uint32_t lo_lead = mapa(smem_u32(const_cast<uint32_t*>(lo_peer)), lead_rank);
    for (int j = 0; j < ntiles; ++j) {
      const int rb = j % kNbuf;
      if (!mbar_wait<false>(bar(bl.ready_local + rb), (j / kNbuf) & 1, status)) break;
      const uint32_t fl = buf_sm + rb * kMsgStride + kFlagOff;
      if ((ld_shared_u32(fl) | ld_shared_u32(fl + 16) | ld_shared_u32(fl + 32) | ld_shared_u32(fl + 48)) != 0)
        st_cluster_u32(lo_lead + 4 * rb, j + 1);
      mbar_arrive_remote(lead(bl.ready + rb));  // release.cluster: the flag and the rescaled O first
    }
  } else if (!is_b && warp >= 4) {
    // ------------------------------------------------------------ pair A: softmax and the messages
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int t = tid - 128;  // TMEM lane
    const int r = t & 63;     // row within this CTA's 64
    const int kh = t >> 6;    // which 64 keys of each tile this thread scores
    const int w = warp - 4;   // its rows' slice: bytes [4096 w, 4096 w + 4096) of P_hi and of P_lo
    const int row = q0 + 64 * static_cast<int>(pr) + r;
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    const uint32_t nb2 = 1 + (w & 1);  // named barrier of warps w and w ^ 2 (lanes t and t ^ 64)
    const float* bias_row = nullptr;
    if (p.bias)
      bias_row = p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(min(row, p.Nq - 1)) * p.bias_sq;
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t s_free_lead0 = lead(bl.s_free), s_free_lead1 = lead(bl.s_free + 1);
    {
      // Q chunks 0 .. kQtc - 1 of this thread's row into its TMEM lane (the TS
      // form's A layout; the threads of lanes r and r + 64 write the same row)
      const uint4* qrow = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q) + b * p.q_sb + h * p.q_sh +
                                                         static_cast<int64_t>(min(row, p.Nq - 1)) * p.q_sn);
      // four chunks' loads in flight before their TMEM stores (a store would
      // otherwise wait for each chunk's global-memory round trip in turn)
#pragma unroll 1
      for (int c0 = 0; c0 < kQtc; c0 += 4) {
        uint4 x[4][8];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int g = 0; g < 8; ++g) x[cc][g] = c0 + cc < kQtc ? __ldg(qrow + 8 * (c0 + cc) + g) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (c0 + cc >= kQtc) break;
          uint32_t wv[32];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            wv[4 * g] = x[cc][g].x;
            wv[4 * g + 1] = x[cc][g].y;
            wv[4 * g + 2] = x[cc][g].z;
            wv[4 * g + 3] = x[cc][g].w;
          }
          tmem_st32(tbase + lane_off + G::kQt + 32 * (c0 + cc), wv);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (pr == 0)
          mbar_arrive(bar(bl.q_full));
        else
          mbar_arrive_remote(lead(bl.q_full));
      }
    }
    bool ok = true;
    float m_used = -INFINITY, l_own = 0.f, l_sum = 0.f;  // l_sum: both halves of the row
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t s_col = (j & 1) ? G::kS1 : G::kS0;
      const int kv0 = j * kTileRows + 64 * kh;  // key of s[0]
      if (bias_row && p.bias_vec) {
        prefetch_l1(bias_row + min(kv0, p.Nkv - 1));
        prefetch_l1(bias_row + min(kv0 + 32, p.Nkv - 1));
        prefetch_l1(bias_row + min(kv0 + 63, p.Nkv - 1));
      }
      const bool got = __all_sync(0xffffffffu, mbar_wait<false>(bar(bl.s_full + (j & 1)), (j >> 1) & 1, status));
      float s[64];
      if (got) {
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tbase + lane_off + s_col, v0);
        tmem_ld32(tbase + lane_off + s_col + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = __uint_as_float(v0[i]);
          s[32 + i] = __uint_as_float(v1[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {  // S_j copied out ("consumed", no data hand-off)
          const uint32_t fr = (j & 1) ? s_free_lead1 : s_free_lead0;
          if (pr == 0)
            mbar_arrive(fr);
          else
            mbar_arrive_remote_relaxed(fr);
        }
      }
      const bool masked = (kv0 + 64 > p.Nkv) || (p.causal && kv0 + 63 > row);
      // scores in the log2 domain: x = s scale log2e (+ bias log2e); without a
      // bias the scale is applied inside the exponent below
      const float c_scale = bias_row ? 1.f : p.scale_log2;
      if (bias_row) {
        if (p.bias_vec && kv0 + 64 <= p.Nkv) {
          const float4* src = reinterpret_cast<const float4*>(bias_row + kv0);
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const float4 x = __ldg(src + g);
            s[4 * g] = fmaf(x.x, kLog2e, s[4 * g] * p.scale_log2);
            s[4 * g + 1] = fmaf(x.y, kLog2e, s[4 * g + 1] * p.scale_log2);
            s[4 * g + 2] = fmaf(x.z, kLog2e, s[4 * g + 2] * p.scale_log2);
            s[4 * g + 3] = fmaf(x.w, kLog2e, s[4 * g + 3] * p.scale_log2);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            s[i] = fmaf(__ldg(bias_row + static_cast<int64_t>(min(kv0 + i, p.Nkv - 1)) * p.bias_sk), kLog2e,
                        s[i] * p.scale_log2);
        }
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
      xmax[t] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c_scale;
      ok = pair_bar_and(nb2, got);  // both warps of the row pair see the same outcome
      if (!ok) break;
      const float m_tile = fmaxf(xmax[t], xmax[t ^ 64]);
      float alpha = 1.f;
      if (m_used == -INFINITY) {
        m_used = m_tile;
      } else if (m_tile > m_used + kRescaleLog2) {
        alpha = ex2(m_used - m_tile);
        m_used = m_tile;
      }
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        s[i] = ex2(fmaf(s[i], c_scale, -m_ref));  // P, in place
        ls[i & 3] += s[i];
      }
      l_own = l_own * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      xsum[t] = l_own;
      pair_bar_and(nb2, true);
      l_sum = xsum[t] + xsum[t ^ 64];
      // the residual term of P on this tile if some row's largest weight
      // exceeds 1/64 of its running sum (this tile included)
      const bool warp_lo = __any_sync(0xffffffffu, ex2(m_tile - m_ref) > kLoFrac * l_sum);
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
      const int rb = j % kNbuf;
      // staging buffer rb: the bulk copies issued from it two tiles ago have read it
      if (lane == 0 && j >= kNbuf) bulk_wait_read<kNbuf - 1>();
      __syncwarp();
      const uint32_t stg = buf_sm + rb * kMsgStride;
      store_row64(stg + kh * kHalfBytes, r, hi);
      store_row64(stg + kPBytes + kh * kHalfBytes, r, lo);
      if (kh == 0) st_shared_v2f(stg + kStatOff + 8 * r, alpha, l_sum);
      if (lane == 0) st_shared_v4(stg + kFlagOff + 16 * w, warp_lo ? 1u : 0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        // pair B's buffer rb is free once its P V products of tile j - 2 are done
        bool fr = true;
        if (j >= kNbuf) fr = mbar_wait<false>(bar(bl.rfree + rb), ((j - kNbuf) / kNbuf) & 1, status);
        if (fr) {
          // pair B's receive buffer rb (its buffers start at offset 0 of its shared memory)
          const uint32_t dst = mapa(base + rb * kMsgStride, other), fb = mapa(bar(bl.rfull + rb), other);
          const uint32_t off = static_cast<uint32_t>(w) * kSlice;
          bulk_copy_s2s(dst + off, stg + off, kSlice, fb);                      // P_hi rows
          bulk_copy_s2s(dst + kPBytes + off, stg + kPBytes + off, kSlice, fb);  // P_lo rows
          if (kh == 0)
            bulk_copy_s2s(dst + kStatOff + 256 * w, stg + kStatOff + 256 * w, 256, fb);  // (alpha, l) of 32 rows
          bulk_copy_s2s(dst + kFlagOff + 16 * w, stg + kFlagOff + 16 * w, 16, fb);      // the residual flag
          bulk_commit_group();
        }
        ok = fr;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
    }
    if (lane == 0) bulk_wait_read<0>();
    // pair B's last commits to each buffer's rfree land here before exit
    if (ok && lane == 0) {
      for (int rb = 0; rb < kNbuf && rb < ntiles && ok; ++rb) {
        const int last = (ntiles - 1 - rb) / kNbuf;
        ok = mbar_wait<false>(bar(bl.rfree + rb), last & 1, status);
      }
    }
    if (kh == 0 && p.lse && row < p.Nq) {
      constexpr float kLn2 = 0.6931471805599453f;
      p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] =
          l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
    }
  } else if (is_b && warp >= 4) {
    // ------------------------------------------------------------ pair B: rescale of O and the epilogue
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int t = tid - 128;  // TMEM lane
    const int r = t & 63;     // row within this CTA's 64
    const int u = t >> 6;     // which half of each O block this lane holds
    const int w = warp - 4;
    const int row = q0 + 64 * static_cast<int>(pr) + r;
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    const uint32_t ready_local = bar(pr == 0 ? bl.ready : bl.ready_local);
    bool ok = true;
    float l_last = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      const int rb = j % kNbuf, use = j / kNbuf;
      ok = __all_sync(0xffffffffu, mbar_wait<false>(bar(bl.rfull + rb), use & 1, status));
      if (!ok) break;
      // no MMA thread waits on this buffer's bytes: warp 0 arms its next use
      if (w == 0 && lane == 0 && j + kNbuf < ntiles) mbar_expect_tx(bar(bl.rfull + rb), kMsgBytes);
      const float2 st = ld_shared_v2f(buf_sm + rb * kMsgStride + kStatOff + 8 * r);  // (alpha, l) of this row
      l_last = st.y;
      if (__any_sync(0xffffffffu, st.x != 1.f) && j > 0) {
        // O *= alpha for this warp's rows, after P_{j-1} V_{j-1} (P_{j+1} V cannot
        // have completed, so the parity is unambiguous)
        ok = __all_sync(0xffffffffu,
                        mbar_wait<false>(bar(bl.pv_done + (j - 1) % kNbuf), ((j - 1) / kNbuf) & 1, status));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4 * kNblk; ++c) {  // this lane's O columns (128 per block)
          uint32_t v[32];
          const uint32_t a = tbase + lane_off + 32 * c;
          tmem_ld32(a, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * st.x);
          tmem_st32(a, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ready_local + 8 * rb);  // release: O rescaled, the message read
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      // the last P V of each buffer (their commits also arrive on the second CTA)
      ok = __all_sync(0xffffffffu,
                      mbar_wait<false>(bar(bl.pv_done + (ntiles - 1) % kNbuf), ((ntiles - 1) / kNbuf) & 1, status));
      if (ok && ntiles >= 2)
        ok = __all_sync(0xffffffffu,
                        mbar_wait<false>(bar(bl.pv_done + (ntiles - 2) % kNbuf), ((ntiles - 2) / kNbuf) & 1, status));
      if (ok) {
        tc_fence_after();
        const float inv_l = l_last > 0.f ? 1.f / l_last : 0.f;
        T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
#pragma unroll 1
        for (int c = 0; c < 4 * kNblk; ++c) {
          // TMEM column 32 c + i of lane 64 u + r: block nb = c / 4, column
          // (N / 2) u + 32 (c mod 4) + i of the block (N = 256, or 128 for a
          // last block of at most 128 columns)
          const int nb = c >> 2, half_n = min(256, G::kD - 256 * nb) > 128 ? 128 : 64;
          const int cc = 32 * (c & 3);
          if (cc >= half_n) continue;
          const int d0 = 256 * nb + half_n * u + cc;
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + 32 * c, v);
          tmem_ld_wait();
          if (row < p.Nq && d0 < G::kD) {
            uint4* dst = reinterpret_cast<uint4*>(orow + d0);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 o;
              o.x = pack2<BF16>(__uint_as_float(v[8 * g + 0]) * inv_l, __uint_as_float(v[8 * g + 1]) * inv_l);
              o.y = pack2<BF16>(__uint_as_float(v[8 * g + 2]) * inv_l, __uint_as_float(v[8 * g + 3]) * inv_l);
              o.z = pack2<BF16>(__uint_as_float(v[8 * g + 4]) * inv_l, __uint_as_float(v[8 * g + 5]) * inv_l);
              o.w = pack2<BF16>(__uint_as_float(v[8 * g + 6]) * inv_l, __uint_as_float(v[8 * g + 7]) * inv_l);
              dst[g] = o;
            }
          }
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

template <int NC, bool BF16>
cudaError_t launch_impl(const FwdParams& p_in, const FwdMaps& m, cudaStream_t st) {
  constexpr int kSmemBytes = Shape<NC>::kSmemBytes;
  FwdParams p = p_in;
  auto kern = fwd_xch_kernel<NC, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * p.q_tiles, p.Hq, p.B);  // (CTA of the cluster, query tile)
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  timing_mark(st);
  e = cudaLaunchKernelEx(&cfg, kern, m.q_half, m.k_half, m.v, p);
  timing_mark(st);
  return e;
}

template <bool BF16>
cudaError_t launch_nc(const FwdParams& p, const FwdMaps& m, cudaStream_t st) {
  switch (p.n_chunks) {
    case 11: return launch_impl<11, BF16>(p, m, st);
    case 12: return launch_impl<12, BF16>(p, m, st);
    case 13: return launch_impl<13, BF16>(p, m, st);
    case 14: return launch_impl<14, BF16>(p, m, st);
    case 15: return launch_impl<15, BF16>(p, m, st);
    case 16: return launch_impl<16, BF16>(p, m, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// D = 576 and 640 stay on the O-split kernel of fwd_fulld.cu: there the
// residual term's extra P V products weigh more than the recomputed S
// (N = 4096, fp16: 0.63 against 0.54 ms), while from D = 704 up this kernel
// is the faster one (D = 1024: 0.80 against 0.87 ms; N = 8192, bf16: 2.68
// against 3.18 ms).
bool fwd_xch_supported(const FwdParams& p) {
  return p.n_chunks >= 11 && p.n_chunks <= 16 && !p.dropout && p.part_o == nullptr;
}

cudaError_t launch_fwd_xch(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_nc<true>(p, m, s) : launch_nc<false>(p, m, s);
}

}  // namespace ffpa
