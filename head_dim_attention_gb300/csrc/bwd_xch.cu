// Attention backward for D = 320..1024 on clusters of four CTAs (two CTA
// pairs) that exchange the probability tiles and their gradients (FFPA
// Attention Benchmark page, "More Benchmark": the SM100 backward's fused
// dK/dV pass, then dQ).  Two modes of one kernel, after the preprocess:
//
//   dK/dV mode (every D), per 128-row key tile, sweeping the query tiles of
//   every query head of the GQA group:
//     pair A: K resident;  X = S^T = K Q^T;  P^T  -> pair B;  dK += dS^T Q
//     pair B: V resident;  X = dP^T = V dO^T; dS^T = P^T (dP^T - Delta) -> A;
//             dV += P^T dO  with P^T straight from the received buffer
//     Separate dV and dK kernels would both rebuild S^T and execute 4 + 6 =
//     10 Nq Nkv D per head; here each pair executes one score product and one
//     gradient product per column tile, 8 Nq Nkv D in all.  A pair cannot hold
//     both gradients (128 x 512 fp32 each takes half of an SM's TMEM in the
//     M = 128 pair layout, and the score tiles need room too), hence the two
//     pairs.  Up to D = 512 one cluster holds all of a gradient's columns;
//     above, two clusters per key tile take one range of columns each (at
//     most 512 wide) and each computes S^T and dP^T over all of D.
//   dQ mode (D = 576..1024, where one pair cannot keep Q and dO resident and
//   hold dQ), per 128-row query tile, sweeping the key tiles:
//     pair A: Q resident;  X = S = Q K^T;  P  -> pair B;
//             dQ[:, columns of A] += dS K  with dS received from B
//     pair B: dO resident; X = dP = dO V^T;  dS = P (dP - Delta) -> A;
//             dQ[:, columns of B] += dS K  with its own dS
//     Each score product is computed once; each pair accumulates one range
//     of dQ's columns.
//
// Layout within a pair (tcgen05 cta_group::2, M = 128): CTA c (c = rank & 1)
// holds stationary rows 64c .. 64c + 63 across all 128 TMEM lanes (lane r:
// row r, the first half of an accumulator's columns; lane r + 64: the second
// half).  CTA r of pair A and CTA r + 2 of pair B hold the same 64 rows; each
// exchange is between those two: every elementwise warp rounds its 32 rows x
// 64 columns of the tile to the input type, writes them into a local staging
// tile in the K-major swizzled operand layout, and copies those 4 KB with one
// bulk copy into the other CTA, whose barrier counts the bytes.  A received
// tile is the receiving pair's A operand as it lies (dK/dV mode: both pairs;
// dQ mode: pair A).  In dQ mode pair B's A operand is its own staging tile.
// Two or three receive buffers per direction cover the round trip (P out, dS
// back) while the score products of the next tiles run.
//
// Signals that cross the two pairs:
//   pt_full[b] / ds_full[b]  bulk-copy bytes, armed by a thread of the
//                            receiving CTA; the second CTA of a pair relays
//                            its completion to the first (pt_peer / ds_peer);
//   pt_free[b]               (in pair A) pair B's elementwise warps have read
//                            the tile (relaxed remote arrives) and, in dK/dV
//                            mode, pair B's dV MMAs have (commit, multicast);
//   ds_free[b]               (in pair B) pair A's gradient commit (multicast).
// In dQ mode pair B's own staging tile is ready once both of its CTAs wrote it
// (st_ready: the second CTA's warps arrive locally and its relay forwards),
// and free once the pair's dQ MMAs and the bulk copy have read it (st_free).
//
// Dropout (philox.cuh; the DROP instantiations): pair A draws the keep bits
// of its scores (in the dK/dV mode with one generator call per lane per eight
// query rows and warp shuffles, since its threads hold key rows) and sends P
// (or P^T) with the sign bit set on dropped entries.  Pair B reads the sign as
// the keep bit and forms dS = P (keep dP / (1 - p) - Delta); in the dK/dV mode
// it then clears the dropped entries of the received tile in place before its
// dV MMAs read it (pm_ready / pm_local, relayed like st_ready), and dV carries
// 1 / (1 - p) in the epilogue.
//
// TMEM per CTA: gradient [0, 256), score tiles [256, 384), the stationary
// tile's chunks 0..3 as the TS-form operand [384, 512) (the score MMAs' operand
// reads from shared memory alone would need the SM's full shared-memory
// bandwidth at M = 128, N = 128).  Warps: 0 producer of the score-operand
// ring (and the stationary tile), 1 TMEM owner + MMA issuer X (first CTA of a
// pair), 2 MMA issuer G (first CTA) or relay (second CTA), 3 producer of the
// gradient-operand ring, 4-7 elementwise, exchange and epilogue.  Every wait
// is bounded (ptx.cuh).
#include <type_traits>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace ffpa {
namespace {

enum Mode : int { kDKV = 0, kDQ = 1 };

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kX0 = 256;               // score buffers at 256 and 320 (64 columns each)
constexpr uint32_t kSt = 384;               // the stationary tile's chunks 0..3 (TS-form A operand)
constexpr int kHalf = kChunkBytes / 2;      // 64 rows x 64 columns, 8 KB
constexpr int kTileX = 2 * kHalf;           // one CTA's exchanged tile: 64 rows x 128 columns, 16 KB
constexpr int kSlice = kTileX / 4;          // one elementwise warp's rows of it, 4 KB
constexpr int kNstage = 2;                  // staging tiles
constexpr int kSlot = 2 * kHalf;            // ring slots of 16 KB
constexpr float kLog2e = 1.4426950408889634f;

template <int NC>
struct Shape {
  static_assert(NC >= 5 && NC <= 16, "D = 320 .. 1024");
  static constexpr int kD = 64 * NC;
  static constexpr int kHalfD = ((kD / 2 + 127) / 128) * 128 < 512 ? ((kD / 2 + 127) / 128) * 128 : 512;
  // dK/dV mode: up to D = 512 one cluster per key tile holds all of a
  // gradient's columns; above, two clusters take [0, kGaKV) and [kGaKV, D)
  static constexpr int kSplitKV = NC <= 8 ? 1 : 2;
  static constexpr int kGaKV = NC <= 8 ? kD : kHalfD;
  // dQ mode: pair A accumulates dQ's columns [0, kGaQ), pair B [kGaQ, D)
  static constexpr int kGaQ = kHalfD;
  static constexpr int kNrecv = NC <= 8 ? 3 : 2;  // receive buffers per direction
  static constexpr int kRes = (NC - 4) * kHalf;  // the stationary tile's chunks 4..NC-1 in shared memory
  static constexpr int kSlots = NC <= 12 ? 3 : 2;  // per ring, as many as fit
  // shared memory: resident | receive buffers | staging | score ring | gradient ring | barriers
  static constexpr int kRecvOff = kRes;
  static constexpr int kStageOff = kRecvOff + kNrecv * kTileX;
  static constexpr int kRingXOff = kStageOff + kNstage * kTileX;
  static constexpr int kRingGOff = kRingXOff + kSlots * kSlot;
  static constexpr int kMiscOff = kRingGOff + kSlots * kSlot;
  static constexpr int kSmemBytes = kMiscOff + 512 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "227 KB per CTA");
  static_assert(kGaKV <= 512 && kD - kGaKV <= 512 && kD - kGaQ <= 512, "ranges of at most 512 columns");
};

struct Bars {
  int full_x, empty_x, full_g, empty_g, res_full, x_full, x_free, pt_full, pt_peer, pt_free, ds_full, ds_peer,
      ds_free, st_ready, st_local, st_free, pm_ready, pm_local, drain_x, drain_g, g_done, count;
};
// rings: up to three slots; x_full, x_free, st_*: one per TMEM score buffer or
// staging tile; pt_*, ds_*, pm_*: one per receive buffer (up to three)
__host__ __device__ constexpr Bars bar_layout() {
  return Bars{0, 3, 6, 9, 12, 13, 15, 17, 20, 23, 26, 29, 32, 35, 37, 39, 41, 44, 47, 48, 49, 50};
}
static_assert(bar_layout().count * 8 + 16 <= 512, "barrier area");

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
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16)
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  else
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Row r of a K-major, 128-byte-swizzled [64 rows x 64 columns] 16-bit subtile:
// granule g (columns 8g .. 8g + 7) at r * 128 + ((g ^ (r & 7)) << 4).
__device__ __forceinline__ uint32_t swz(uint32_t tile, int r, int g) {
  return tile + static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(g) ^ static_cast<uint32_t>(r & 7)) << 4);
}

// Geometry of a cluster: its stationary tile, gradient range and column sweep.
struct Geo {
  int b, hs, kvh;      // batch, head of the stationary tensor, kv head
  int st, s_row0;      // stationary tile; this CTA's first stationary row
  int s_limit;         // rows of the stationary tensor
  int g0, gw;          // this CTA's gradient columns [g0, g0 + gw)
  int nv0, nv1;        // 64-column chunks per CTA of the gradient's two halves (N = 128 nv)
  int qt_begin, nq_h;  // dK/dV mode: first query tile and query tiles per head
  int ncols, rot;      // column tiles and the sweep's start
};

template <int MODE, int NC>
__device__ __forceinline__ Geo make_geo(const BwdParams& p, int pr, bool is_b) {
  using G = Shape<NC>;
  Geo g;
  g.b = blockIdx.z;
  const int cl = static_cast<int>(blockIdx.x) >> 2;
  int gsel;
  if (MODE == kDKV) {
    gsel = G::kSplitKV == 2 ? (cl & 1) : 0;  // above D = 512 two clusters per key tile
    g.st = cl / G::kSplitKV;
    g.kvh = blockIdx.y;
    g.hs = g.kvh;
    g.s_limit = p.Nkv;
    g.qt_begin = p.causal ? g.st : 0;  // top-left causal: query rows i >= key row j
    g.nq_h = max(0, p.q_tiles - g.qt_begin);
    g.ncols = p.group * g.nq_h;
  } else {
    gsel = is_b ? 1 : 0;  // each pair accumulates one range of dQ's columns
    g.st = p.q_tiles - 1 - cl;  // heavy causal tiles first
    g.hs = blockIdx.y;
    g.kvh = g.hs / p.group;
    g.s_limit = p.Nq;
    const int kv_end = p.causal ? min(p.Nkv, (g.st + 1) * kTileRows) : p.Nkv;
    g.ncols = (kv_end + kTileRows - 1) / kTileRows;
    g.qt_begin = 0;
    g.nq_h = 0;
  }
  const int ga = MODE == kDKV ? G::kGaKV : G::kGaQ;
  g.g0 = gsel ? ga : 0;
  g.gw = gsel ? G::kD - ga : ga;
  g.nv0 = g.gw >= 256 ? 2 : (g.gw + 127) / 128;
  g.nv1 = g.gw > 256 ? (g.gw - 256 + 127) / 128 : 0;
  g.s_row0 = g.st * kTileRows + 64 * pr;
  g.rot = g.ncols > 0 ? g.st % g.ncols : 0;
  return g;
}

// Column tile c: head of the column tensor and its first row.
template <int MODE>
__device__ __forceinline__ void column(const Geo& g, const BwdParams& p, int c, int* head, int* row0) {
  c += g.rot;
  if (c >= g.ncols) c -= g.ncols;
  if (MODE == kDKV) {
    *head = g.kvh * p.group + c / g.nq_h;
    *row0 = (g.qt_begin + c % g.nq_h) * kTileRows;
  } else {
    *head = g.kvh;
    *row0 = c * kTileRows;
  }
}

template <int MODE, int NC, bool BF16, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_xch_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                   const __grid_constant__ CUtensorMap map_vh, const __grid_constant__ CUtensorMap map_doh,
                   const __grid_constant__ BwdParams p) {
  using G = Shape<NC>;
  constexpr int kSlots = G::kSlots, kNrecv = G::kNrecv;
  constexpr bool DQ = MODE == kDQ;
  constexpr Bars bl = bar_layout();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t res_sm = smem_u32(smem), recv_sm = res_sm + G::kRecvOff, stage_sm = res_sm + G::kStageOff;
  const uint32_t ring_x = res_sm + G::kRingXOff, ring_g = res_sm + G::kRingGOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0, 1: pair A; 2, 3: pair B
  const bool is_b = rank >= 2;
  const uint32_t pr = rank & 1, lead_rank = rank & 2, other = rank ^ 2;  // other: same rows, other pair
  const uint16_t pair_mask = static_cast<uint16_t>(3u << lead_rank);
  const uint16_t other_mask = static_cast<uint16_t>(3u << (lead_rank ^ 2));
  const Geo g = make_geo<MODE, NC>(p, static_cast<int>(pr), is_b);
  uint32_t* status = p.status;
  auto lead = [&](int i) { return pr == 0 ? bar(i) : mapa(bar(i), lead_rank); };
  // pair B's gradient operand in dQ mode is its own staging tile
  const bool own_operand = DQ && is_b;

  // stationary tile, score-product column operand (K-major), gradient column operand (MN-major)
  const CUtensorMap* mRes = DQ ? (is_b ? &map_doh : &map_qh) : (is_b ? &map_vh : &map_kh);
  const CUtensorMap* mX = DQ ? (is_b ? &map_vh : &map_kh) : (is_b ? &map_doh : &map_qh);
  const CUtensorMap* mG = DQ ? &map_kh : (is_b ? &map_doh : &map_qh);

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar(bl.full_x + i), 1);
      mbar_init(bar(bl.empty_x + i), 1);
      mbar_init(bar(bl.full_g + i), 1);
      mbar_init(bar(bl.empty_g + i), 1);
    }
    // stationary tile ready: the armed TMA bytes (chunks 4..NC-1) and the eight
    // elementwise warps of the pair that wrote chunks 0..3 into TMEM
    mbar_init(bar(bl.res_full), 1 + 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.x_full + i), 1);
      mbar_init(bar(bl.x_free + i), 8);  // four elementwise warps in each CTA of the pair
      mbar_init(bar(bl.st_ready + i), 5);  // dQ mode, pair B: four local warps + the second CTA's relay
      mbar_init(bar(bl.st_local + i), 4);  // (second CTA) its four elementwise warps
      mbar_init(bar(bl.st_free + i), 1);   // the pair's dQ commit
    }
    for (int i = 0; i < kNrecv; ++i) {
      mbar_init(bar(bl.pt_full + i), 1);
      mbar_init(bar(bl.pt_peer + i), 1);
      mbar_init(bar(bl.pt_free + i), DQ ? 4 : 5);  // the other CTA's four warps (+ pair B's dV commit)
      mbar_init(bar(bl.ds_full + i), 1);
      mbar_init(bar(bl.ds_peer + i), 1);
      mbar_init(bar(bl.ds_free + i), 1);  // pair A's gradient commit
      mbar_init(bar(bl.pm_ready + i), 5);  // dropout, dK/dV mode, pair B: four local warps + the relay
      mbar_init(bar(bl.pm_local + i), 4);  // (second CTA) its four elementwise warps
    }
    mbar_init(bar(bl.drain_x), 1);
    mbar_init(bar(bl.drain_g), 1);
    mbar_init(bar(bl.g_done), 1);
    // the first use of each receive buffer: this CTA expects one tile's bytes
    for (int i = 0; i < kNrecv; ++i) mbar_expect_tx(bar((is_b ? bl.pt_full : bl.ds_full) + i), kTileX);
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
  const int ncols = g.ncols;
  const int nhalves = g.nv1 > 0 ? 2 : 1;

  if ((warp == 0 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ TMA producers (X ring: warp 0, G ring: warp 3)
    // The bytes of both CTAs' loads are counted on the first CTA's full barrier.
    const bool is_x = warp == 0;
    const int full0 = is_x ? bl.full_x : bl.full_g, empty0 = is_x ? bl.empty_x : bl.empty_g;
    const uint32_t ring = is_x ? ring_x : ring_g;
    if (is_x) {
      tma_prefetch_desc(mRes);
      tma_prefetch_desc(mX);
      if (pr == 0) mbar_expect_tx(bar(bl.res_full), 2 * G::kRes);
      for (int c = 4; c < NC; ++c)
        tma_load_4d_pair(res_sm + (c - 4) * kHalf, mRes, lead(bl.res_full), c * kChunk, g.s_row0, g.hs, g.b);
    } else {
      tma_prefetch_desc(mG);
    }
    bool ok = true;
    uint32_t it = 0;
    auto next_slot = [&](uint32_t* dst, uint32_t* fb, int bytes) -> bool {
      const uint32_t s = it % kSlots, r = it / kSlots;
      ++it;
      if (!mbar_wait(bar(empty0 + s), (r & 1) ^ 1, status)) return false;
      *dst = ring + s * kSlot;
      *fb = lead(full0 + s);
      if (pr == 0) mbar_expect_tx(bar(full0 + s), 2 * bytes);
      return true;
    };
    for (int c = 0; c < ncols && ok; ++c) {
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      if (is_x) {
        // this CTA's 64 column rows over all of D, two chunks per slot
        for (int x = 0; x < NC && ok; x += 2) {
          const int n = min(2, NC - x);
          uint32_t dst, fb;
          if (!(ok = next_slot(&dst, &fb, n * kHalf))) break;
          for (int i = 0; i < n; ++i)
            tma_load_4d_pair(dst + i * kHalf, mX, fb, (x + i) * kChunk, cr0 + 64 * static_cast<int>(pr), ch, g.b);
        }
      } else {
        // gradient operand: for each half h of this CTA's gradient columns and
        // each 64-row half kh of the column tile, this CTA's one or two chunks
        for (int h = 0; h < nhalves && ok; ++h) {
          const int nv = h == 0 ? g.nv0 : g.nv1;
          for (int kh = 0; kh < 2 && ok; ++kh) {
            uint32_t dst, fb;
            if (!(ok = next_slot(&dst, &fb, nv * kHalf))) break;
            for (int i = 0; i < nv; ++i)
              tma_load_4d_pair(dst + i * kHalf, mG, fb, g.g0 + (4 * h + nv * static_cast<int>(pr) + i) * kChunk,
                               cr0 + 64 * kh, ch, g.b);
          }
        }
      }
    }
    // the ring's last commits (they arrive on both CTAs) complete before exit
    for (uint32_t s = 0; s < static_cast<uint32_t>(kSlots) && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / kSlots) * kSlots;
      mbar_wait(bar(empty0 + s), (last / kSlots) & 1, status);
    }
  } else if (warp == 1 && lane == 0 && pr == 0) {
    // ------------------------------------------------------------ MMA issuer X: score product of each column tile
    constexpr uint32_t idesc_x = idesc_f16(BF16, 128, 128, false, false);  // 128 stationary rows x 128 columns
    const uint64_t dres = sdesc_sw128(res_sm, 16, 1024);
    const uint64_t dring = sdesc_sw128(ring_x, 16, 1024);
    constexpr int kSlotsPerTile = (NC + 1) / 2;
    constexpr bool kRagged = (NC & 1) != 0;
    bool ok = mbar_wait(bar(bl.res_full), 0, status);
    tc_fence_after();
    uint32_t it = 0;
    for (int c = 0; c < ncols && ok; ++c) {
      if (c >= 2) {
        // the elementwise warps of both CTAs have copied X_{c-2} out of this buffer
        ok = mbar_wait(bar(bl.x_free + (c & 1)), ((c - 2) >> 1) & 1, status);
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t x_tm = tbase + kX0 + 64 * (c & 1);
      for (int m = 0; m < kSlotsPerTile && ok; ++m) {
        const uint32_t s = it % kSlots;
        ok = mbar_wait(bar(bl.full_x + s), (it / kSlots) & 1, status);
        ++it;
        if (!ok) break;
        tc_fence_after();
        const uint64_t bs = sdesc_advance(dring, s * kSlot);
        if (m < 2) {  // chunks 0..3: the stationary tile from TMEM (8 columns per 16-column step)
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint64_t bd = sdesc_advance(bs, i * kHalf);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ts_pair(x_tm, tbase + kSt + 32 * (2 * m + i) + 8 * kk, sdesc_advance(bd, kk * 32), idesc_x,
                           (m | i | kk) != 0);
          }
        } else {  // chunks 4..NC-1 from shared memory
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (kRagged && 2 * m + i >= NC) break;
            const uint64_t a = sdesc_advance(dres, (2 * m + i - 4) * kHalf);
            const uint64_t bd = sdesc_advance(bs, i * kHalf);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_pair(x_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x, 1u);
          }
        }
        umma_commit_pair(bar(bl.empty_x + s), pair_mask);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.x_full + (c & 1)), pair_mask);
    }
    umma_commit_pair(bar(bl.drain_x), static_cast<uint16_t>(1u << rank));
    mbar_wait(bar(bl.drain_x), 0, status);
  } else if (warp == 2 && lane == 0 && pr == 0) {
    // ------------------------------------------------------------ MMA issuer G: gradient += (received or own tile) x column operand
    constexpr uint32_t idesc_g256 = idesc_f16(BF16, 128, 256, false, true);  // stationary rows x 256 columns
    constexpr uint32_t idesc_g128 = idesc_f16(BF16, 128, 128, false, true);
    const uint64_t dring = sdesc_sw128(ring_g, kHalf, 1024);  // MN-major: 64-column atoms 8 KB apart
    const uint64_t drecv = sdesc_sw128(recv_sm, 16, 1024);   // received tile, K-major
    const uint64_t dstage = sdesc_sw128(stage_sm, 16, 1024);  // own staging tile (dQ mode, pair B)
    const int rfull = is_b ? bl.pt_full : bl.ds_full, rpeer = is_b ? bl.pt_peer : bl.ds_peer;
    const int rfree = is_b ? bl.pt_free : bl.ds_free;
    bool ok = true;
    uint32_t it = 0;
    for (int c = 0; c < ncols && ok; ++c) {
      const int rb = c % kNrecv, use = c / kNrecv;
      uint64_t da;
      if (own_operand) {
        // both CTAs' elementwise warps have written their dS into staging tile c mod 2
        ok = mbar_wait(bar(bl.st_ready + (c & 1)), (c >> 1) & 1, status);
        if (!ok) break;
        da = sdesc_advance(dstage, (c % kNstage) * kTileX);
      } else {
        // this CTA's and the second CTA's halves of the tile have arrived
        ok = mbar_wait(bar(rfull + rb), use & 1, status);
        if (!ok) break;
        if (c + kNrecv < ncols) mbar_expect_tx(bar(rfull + rb), kTileX);  // the buffer's next use
        ok = mbar_wait(bar(rpeer + rb), use & 1, status);
        if (!ok) break;
        if (DROP && !DQ && is_b) {
          // dropout: both CTAs' elementwise warps have zeroed the dropped P^T entries in place
          ok = mbar_wait(bar(bl.pm_ready + rb), use & 1, status);
          if (!ok) break;
        }
        da = sdesc_advance(drecv, rb * kTileX);
      }
      tc_fence_after();
      for (int h = 0; h < nhalves && ok; ++h) {
        const uint32_t acc_tm = tbase + 128 * h;
        const uint32_t idg = (h == 0 ? g.nv0 : g.nv1) == 2 ? idesc_g256 : idesc_g128;
        for (int kh = 0; kh < 2 && ok; ++kh) {
          const uint32_t s = it % kSlots;
          ok = mbar_wait(bar(bl.full_g + s), (it / kSlots) & 1, status);
          ++it;
          if (!ok) break;
          tc_fence_after();
          const uint64_t bs = sdesc_advance(dring, s * kSlot);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)  // 16-row steps: A subtile kh, B slot rows 16 k4 ..
            umma_ss_pair(acc_tm, sdesc_advance(da, kh * kHalf + k4 * 32), sdesc_advance(bs, k4 * 2048), idg,
                         (c > 0 || kh > 0 || k4 > 0) ? 1u : 0u);
          umma_commit_pair(bar(bl.empty_g + s), pair_mask);
        }
      }
      if (!ok) break;
      if (own_operand)
        umma_commit_pair(bar(bl.st_free + (c & 1)), pair_mask);  // the staging tile may be rewritten
      else if (!(DQ && is_b))
        umma_commit_pair(bar(rfree + rb), other_mask);  // the received buffer may be refilled
    }
    if (ncols > 0) umma_commit_pair(bar(bl.g_done), pair_mask);  // the epilogue waits it only then
    umma_commit_pair(bar(bl.drain_g), static_cast<uint16_t>(1u << rank));
    mbar_wait(bar(bl.drain_g), 0, status);
  } else if (warp == 2 && lane == 0 && pr == 1) {
    // ------------------------------------------------------------ relay for the pair's first CTA
    if (own_operand) {
      // dQ mode, pair B: this CTA's dS staging tile is written
      for (int c = 0; c < ncols; ++c) {
        if (!mbar_wait(bar(bl.st_local + (c & 1)), (c >> 1) & 1, status)) break;
        mbar_arrive_remote(lead(bl.st_ready + (c & 1)));  // release.cluster: the tile is visible first
      }
    } else {
      const int rfull = is_b ? bl.pt_full : bl.ds_full, rpeer = is_b ? bl.pt_peer : bl.ds_peer;
      for (int c = 0; c < ncols; ++c) {
        const int rb = c % kNrecv, use = c / kNrecv;
        if (!mbar_wait(bar(rfull + rb), use & 1, status)) break;
        if (c + kNrecv < ncols) mbar_expect_tx(bar(rfull + rb), kTileX);
        mbar_arrive_remote(lead(rpeer + rb));  // release.cluster: the tile is visible to the first CTA's MMAs
        if (DROP && !DQ && is_b) {  // and, with dropout, once this CTA's warps have masked it
          if (!mbar_wait(bar(bl.pm_local + rb), use & 1, status)) break;
          mbar_arrive_remote(lead(bl.pm_ready + rb));
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise, exchange, epilogue
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int t = tid - 128;  // TMEM lane
    const int r = t & 63;     // stationary row within this CTA's 64
    const int u = t >> 6;     // column half of the column tile
    const int w = warp - 4;   // rows 32 (w & 1) .. of column half w >> 1: bytes [4096 w, 4096 w + 4096) of a tile
    const int srow = g.s_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
    // the other pair's CTA that holds the same rows receives this side's tiles
    const int o_full = is_b ? bl.ds_full : bl.pt_full;
    const int sfree = is_b ? bl.ds_free : bl.pt_free;  // this side's "the other's buffer is free"
    {
      // chunks 0..3 of this thread's stationary row into its TMEM lane: 128
      // words of two 16-bit values in memory order, the TS form's A layout
      // (the threads of lanes r and r + 64 write the same row)
      const T* base;
      int64_t sb, sh, sn;
      if (DQ) {
        base = reinterpret_cast<const T*>(is_b ? p.dout : p.q);
        sb = is_b ? p.do_sb : p.q_sb; sh = is_b ? p.do_sh : p.q_sh; sn = is_b ? p.do_sn : p.q_sn;
      } else {
        base = reinterpret_cast<const T*>(is_b ? p.v : p.k);
        sb = is_b ? p.v_sb : p.k_sb; sh = is_b ? p.v_sh : p.k_sh; sn = is_b ? p.v_sn : p.k_sn;
      }
      const uint4* srow_ptr = reinterpret_cast<const uint4*>(base + g.b * sb + g.hs * sh +
                                                             static_cast<int64_t>(min(srow, g.s_limit - 1)) * sn);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t wv[32];
#pragma unroll
        for (int gq = 0; gq < 8; ++gq) {
          const uint4 x = __ldg(srow_ptr + 8 * c + gq);
          wv[4 * gq] = x.x;
          wv[4 * gq + 1] = x.y;
          wv[4 * gq + 2] = x.z;
          wv[4 * gq + 3] = x.w;
        }
        tmem_st32(tbase + lane_off + kSt + 32 * c, wv);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (pr == 0)
          mbar_arrive(bar(bl.res_full));
        else
          mbar_arrive_remote(lead(bl.res_full));
      }
    }
    // dQ mode: the row statistics of this thread's query row
    float row_stat = 0.f;
    if (DQ) {
      const int64_t idx = (static_cast<int64_t>(g.b) * p.Hq + g.hs) * p.Nq + min(srow, p.Nq - 1);
      row_stat = is_b ? p.delta[idx] : p.lse2[idx];
    }
    // dK/dV mode: column statistics of a column tile; lane l holds those of
    // query rows cbase + l and cbase + 32 + l.  They are loaded one column tile
    // ahead, so that the loads are in flight during the score product.
    const float* stat_vec = is_b ? p.delta : p.lse2;
    auto load_stats = [&](int c, float (&dst)[2]) {
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      const int64_t sbase = (static_cast<int64_t>(g.b) * p.Hq + ch) * p.Nq;
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) dst[k2] = stat_vec[sbase + min(cr0 + 64 * u + 32 * k2 + lane, p.Nq - 1)];
    };
    float cs_next[2] = {0.f, 0.f};
    if (!DQ && ncols > 0) load_stats(0, cs_next);
    bool ok = true;
    for (int c = 0; c < ncols; ++c) {
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      const int cbase = cr0 + 64 * u;  // first column row of this thread's half
      const int rb = c % kNrecv, use = c / kNrecv;
      float cs[2] = {cs_next[0], cs_next[1]};
      if (!DQ && c + 1 < ncols) load_stats(c + 1, cs_next);
      // statistic of column e of this thread's half (per query row: the column
      // in dK/dV mode, this thread's row in dQ mode)
      auto stat = [&](int e) { return DQ ? row_stat : __shfl_sync(0xffffffffu, cs[e >> 5], e & 31); };
      // dropout, pair A: the keep bits of this thread's 64 scores (query head
      // hs in dQ mode, the column's query head in dK/dV mode), drawn while the
      // score product runs; bit e for column e
      uint32_t keep_lo = 0, keep_hi = 0;
      if constexpr (DROP) {
        if (!is_b) {
          DropKey dk = {p.drop_seed_lo, p.drop_seed_hi, static_cast<uint32_t>(g.b * p.Hq + (DQ ? g.hs : ch)),
                        p.drop_off, p.drop_t};
          if (DQ)
            keep64_row(dk, cbase, srow, keep_lo, keep_hi);
          else
            keep64_col(dk, g.s_row0 + 32 * (w & 1), cbase, lane, keep_lo, keep_hi);
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x_full + (c & 1)), (c >> 1) & 1, status));
      if (!ok) break;
      tc_fence_after();
      float xv[64];
      {
        uint32_t a0[32], a1[32];
        const uint32_t col = kX0 + 64 * (c & 1);
        tmem_ld32(tbase + lane_off + col, a0);
        tmem_ld32(tbase + lane_off + col + 32, a1);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          xv[e] = __uint_as_float(a0[e]);
          xv[32 + e] = __uint_as_float(a1[e]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // X consumed (no data hand-off)
        if (pr == 0)
          mbar_arrive(bar(bl.x_free + (c & 1)));
        else
          mbar_arrive_remote_relaxed(lead(bl.x_free + (c & 1)));
      }
      uint32_t wds[32];
      if (!is_b) {
        // P (dQ mode: query row srow, keys cbase..) or P^T (dK/dV mode: key row
        // srow, queries cbase..) = 2^(S scale log2e + bias log2e - lse2), 0 where masked
        bool plain;
        if (DQ)
          plain = srow < p.Nq && cbase + 64 <= p.Nkv && (!p.causal || cbase + 63 <= srow) && row_stat > -INFINITY;
        else
          plain = srow < p.Nkv && cbase + 64 <= p.Nq && (!p.causal || srow <= cbase);
        plain = __all_sync(0xffffffffu, plain) && p.bias == nullptr;
        if (plain) {
#pragma unroll
          for (int e = 0; e < 64; ++e) xv[e] = ex2(fmaf(xv[e], p.scale_log2, -stat(e)));
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int i = DQ ? srow : cbase + e, j = DQ ? cbase + e : srow;  // query row, key
            const float l2 = stat(e);
            const bool valid = i < p.Nq && j < p.Nkv && !(p.causal && j > i) && l2 > -INFINITY;
            float xx = fmaf(xv[e], p.scale_log2, -l2);
            if (p.bias)
              xx = fmaf(__ldg(p.bias + g.b * p.bias_sb + (DQ ? g.hs : ch) * p.bias_sh +
                              static_cast<int64_t>(min(i, p.Nq - 1)) * p.bias_sq +
                              static_cast<int64_t>(min(j, p.Nkv - 1)) * p.bias_sk),
                        kLog2e, xx);
            xv[e] = valid ? ex2(xx) : 0.f;
          }
        }
        if constexpr (DROP) {
          // a dropped probability travels with its sign bit set
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (!(((e < 32 ? keep_lo : keep_hi) >> (e & 31)) & 1u)) xv[e] = -xv[e];
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) wds[e] = pack2<BF16>(xv[2 * e], xv[2 * e + 1]);
      } else {
        // dS = P (dP - Delta), P from pair A's tile
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.pt_full + rb), use & 1, status));
        if (!ok) break;
        // dQ mode: no MMA thread waits on this buffer, so warp 0 arms its next use
        if (DQ && w == 0 && lane == 0 && c + kNrecv < ncols) mbar_expect_tx(bar(bl.pt_full + rb), kTileX);
        const uint32_t pt = recv_sm + rb * kTileX + u * kHalf;
#pragma unroll
        for (int gq = 0; gq < 8; ++gq) {
          const uint4 v = ld_shared_v4(swz(pt, r, gq));
          const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
          uint32_t pm[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = 8 * gq + 2 * q;
            if constexpr (DROP) {
              // dropout: the sign bit marks a dropped probability; dP of the
              // dropped output is dO V^T times keep / (1 - p)
              const uint32_t wq = pw[q];
              const float2 pp = unpack2<BF16>(wq & 0x7FFF7FFFu);
              const float d0 = (wq & 0x8000u) ? 0.f : xv[e] * p.drop_scale;
              const float d1 = (wq & 0x80000000u) ? 0.f : xv[e + 1] * p.drop_scale;
              wds[4 * gq + q] = pack2<BF16>(pp.x * (d0 - stat(e)), pp.y * (d1 - stat(e + 1)));
              pm[q] = wq & ~(((wq >> 15) & 0x00010001u) * 0xFFFFu);  // dropped entries -> +0
            } else {
              const float2 pp = unpack2<BF16>(pw[q]);
              wds[4 * gq + q] = pack2<BF16>(pp.x * (xv[e] - stat(e)), pp.y * (xv[e + 1] - stat(e + 1)));
              pm[q] = 0u;
            }
          }
          // dK/dV mode with dropout: dV's MMAs read P^T with the dropped entries zeroed
          if (DROP && !DQ) st_shared_v4(swz(pt, r, gq), pm[0], pm[1], pm[2], pm[3]);
        }
        if (DROP && !DQ) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar((pr == 0 ? bl.pm_ready : bl.pm_local) + rb));
        }
        __syncwarp();
        // P has been read into registers: pair A may refill this buffer once
        // (dK/dV mode) the dV MMAs have read it too (their commit is the fifth arrive)
        if (lane == 0) mbar_arrive_remote_relaxed(mapa(bar(bl.pt_free + rb), other));
      }
      // staging tile c mod 2: the bulk copy issued from it two tiles ago has read
      // it, and (dQ mode, pair B) so have the pair's dQ MMAs of that tile
      if (lane == 0 && c >= kNstage) bulk_wait_read<kNstage - 1>();
      if (own_operand && c >= kNstage) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.st_free + (c & 1)), ((c - 2) >> 1) & 1, status));
        if (!ok) break;
      }
      __syncwarp();
      {
        const uint32_t st = stage_sm + (c % kNstage) * kTileX + u * kHalf;
#pragma unroll
        for (int gq = 0; gq < 8; ++gq)
          st_shared_v4(swz(st, r, gq), wds[4 * gq], wds[4 * gq + 1], wds[4 * gq + 2], wds[4 * gq + 3]);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (own_operand && lane == 0) mbar_arrive(bar((pr == 0 ? bl.st_ready : bl.st_local) + (c & 1)));
      if (lane == 0) {
        // the other pair's buffer rb is free once its use c - kNrecv is finished
        bool fr = true;
        if (c >= kNrecv) fr = mbar_wait(bar(sfree + rb), (use - 1) & 1, status);
        if (fr) {
          const uint32_t off = static_cast<uint32_t>(w) * kSlice;
          bulk_copy_s2s(mapa(recv_sm + rb * kTileX + off, other), stage_sm + (c % kNstage) * kTileX + off, kSlice,
                        mapa(bar(o_full + rb), other));
          bulk_commit_group();
        }
        ok = fr;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
    }
    if (lane == 0) bulk_wait_read<0>();
    // the other pair's last frees of each buffer (its commits and arrives land here)
    if (ok && lane == 0) {
      for (int rb = 0; rb < kNrecv && rb < ncols && ok; ++rb) {
        const int last = (ncols - 1 - rb) / kNrecv;
        ok = mbar_wait(bar(sfree + rb), last & 1, status);
      }
    }
    // dQ mode, pair B: the last dQ commits on the staging tiles
    if (own_operand && ok && lane == 0) {
      for (int sb = 0; sb < kNstage && sb < ncols && ok; ++sb) {
        const int last = (ncols - 1 - sb) / kNstage;
        ok = mbar_wait(bar(bl.st_free + sb), last & 1, status);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
      // ---------------------------------------------------------- epilogue
      if (ncols > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.g_done), 0, status));
        tc_fence_after();
      }
      if (ok) {
        T* dst_base;
        int64_t sb, sh, sn;
        if (DQ) {
          dst_base = reinterpret_cast<T*>(p.dq); sb = p.dq_sb; sh = p.dq_sh; sn = p.dq_sn;
        } else if (is_b) {
          dst_base = reinterpret_cast<T*>(p.dv); sb = p.dv_sb; sh = p.dv_sh; sn = p.dv_sn;
        } else {
          dst_base = reinterpret_cast<T*>(p.dk); sb = p.dk_sb; sh = p.dk_sh; sn = p.dk_sn;
        }
        const float mul = (!DQ && is_b) ? (DROP ? p.drop_scale : 1.f) : p.scale;  // dV: kept P carries 1 / (1 - p)
        T* orow = dst_base + g.b * sb + g.hs * sh + static_cast<int64_t>(srow) * sn;
        const int gcols = 128 + 64 * g.nv1;  // TMEM columns of the gradient per lane
        for (int k = 0; k < gcols / 32; ++k) {
          // TMEM column 32 k of lane 64 u + r: half 0 (k < 4) is gradient column
          // g0 + 64 nv0 u + 32 k, half 1 is g0 + 256 + 64 nv1 u + 32 (k - 4)
          int dcol;
          if (k < 4)
            dcol = k < 2 * g.nv0 ? g.g0 + 64 * g.nv0 * u + 32 * k : G::kD;
          else
            dcol = k - 4 < 2 * g.nv1 ? g.g0 + 256 + 64 * g.nv1 * u + 32 * (k - 4) : G::kD;
          uint32_t v[32];
          if (ncols > 0) {
            tmem_ld32(tbase + lane_off + 32 * k, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (srow < g.s_limit && dcol < G::kD) {
            uint4* dst = reinterpret_cast<uint4*>(orow + dcol);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 o;
              o.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]) * mul, __uint_as_float(v[8 * q4 + 1]) * mul);
              o.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]) * mul, __uint_as_float(v[8 * q4 + 3]) * mul);
              o.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]) * mul, __uint_as_float(v[8 * q4 + 5]) * mul);
              o.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]) * mul, __uint_as_float(v[8 * q4 + 7]) * mul);
              dst[q4] = o;
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

template <int MODE, int NC, bool BF16>
cudaError_t launch_impl(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  constexpr int smem = Shape<NC>::kSmemBytes;
  auto kern = p.dropout ? bwd_xch_kernel<MODE, NC, BF16, true> : bwd_xch_kernel<MODE, NC, BF16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // dK/dV: one or two clusters per key tile (one per range of gradient columns); dQ: one per query tile
  cfg.gridDim = MODE == kDKV ? dim3(4 * Shape<NC>::kSplitKV * p.kv_tiles, p.Hkv, p.B) : dim3(4 * p.q_tiles, p.Hq, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, m.q_half, m.k_half, m.v_half, m.dout_half, p);
  timing_mark(st);
  return e;
}

template <int MODE, bool BF16>
cudaError_t launch_nc(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  if constexpr (MODE == kDKV) {
    switch (p.n_chunks) {
      case 5: return launch_impl<MODE, 5, BF16>(p, m, st);
      case 6: return launch_impl<MODE, 6, BF16>(p, m, st);
      case 7: return launch_impl<MODE, 7, BF16>(p, m, st);
      case 8: return launch_impl<MODE, 8, BF16>(p, m, st);
      default: break;
    }
  }
  switch (p.n_chunks) {
    case 9: return launch_impl<MODE, 9, BF16>(p, m, st);
    case 10: return launch_impl<MODE, 10, BF16>(p, m, st);
    case 11: return launch_impl<MODE, 11, BF16>(p, m, st);
    case 12: return launch_impl<MODE, 12, BF16>(p, m, st);
    case 13: return launch_impl<MODE, 13, BF16>(p, m, st);
    case 14: return launch_impl<MODE, 14, BF16>(p, m, st);
    case 15: return launch_impl<MODE, 15, BF16>(p, m, st);
    case 16: return launch_impl<MODE, 16, BF16>(p, m, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool bwd_xch_dkv_supported(const BwdParams& p) { return p.n_chunks >= 5 && p.n_chunks <= 16; }
bool bwd_xch_dq_supported(const BwdParams& p) { return p.n_chunks >= 9 && p.n_chunks <= 16; }

cudaError_t launch_bwd_xch_dkv(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_nc<kDKV, true>(p, m, s) : launch_nc<kDKV, false>(p, m, s);
}
cudaError_t launch_bwd_xch_dq(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_nc<kDQ, true>(p, m, s) : launch_nc<kDQ, false>(p, m, s);
}

}  // namespace ffpa
