// Attention backward dQ for D = 320..512, the third launch after the
// preprocess and the fused dK/dV kernel of bwd_xch.cu (FFPA Attention
// Benchmark page, "More Benchmark": the SM100 backward's separate dQ pass).
// P is rebuilt from the forward's lse; per 128-row query tile, over the key
// tiles (to the diagonal when causal):
//   S = Q K^T, dP = dO V^T, dS = P (dP - Delta),  dQ += dS K  (3 GEMMs)
// and dQ is scaled by `scale` in the epilogue.
//
// Why M = 128 pairs.  A 128 x 512 fp32 gradient fills a CTA's 512 TMEM
// columns, so a one-CTA kernel (or an M = 256 pair) must split the gradient's
// columns over CTAs that each recompute S and dP over the whole of D.  With
// cta_group::2 and M = 128 each SM holds 64 rows of the accumulator across all
// 128 TMEM lanes (lane r: row r, the first N/2 columns; lane r + 64: row r,
// the other N/2), so the 128 x D gradient of a query tile takes at most 256
// columns per SM and S and dP are computed once.
//
// Per pair: CTA c holds query rows 64c .. 64c + 63 of the tile and keeps Q and
// dO resident in shared memory (64 rows x D each).  The kernel sweeps 128-row
// key tiles.  Per key tile:
//   X1 = S         M=128, N=128 (B split by N: CTA c loads keys 64c ..),
//                  reduced over the NC 64-column chunks of D
//   X2 = dP        the same with dO and V
//   dS             elementwise, rounded to the input type, written to shared
//                  memory as the K-major A operand (64 rows x 128 keys), in
//                  two buffers used by alternate key tiles, so the
//                  elementwise warps write one while the dQ MMAs read the other
//   dQ             ceil(NC / 2) quarters of 128 columns, M=128, N=128: CTA c
//                  supplies the 64 columns 128 qd + 64 c .. of K (MN-major);
//                  columns past D are zero-filled by TMA and not stored
// Each of these pair MMAs costs the issuing thread more time than the tensor
// core needs for it, and each barrier wait costs it about as much as four
// MMAs, so one thread cannot keep the tensor core busy.  Two threads issue:
//   thread A: S and dQ quarters 0, 1;  thread B: dP and the other quarters.
// Each issuing thread has its own ring of two 16 KB slots with its own TMA
// producer, so every ring keeps a single producer and a single consumer.
// (Q's first chunks in TMEM as the TS operand, or dQ in two N = 256 halves,
// both measured slower here than this layout.)
//
// Signals from the second CTA of the pair to the first: "X consumed" is a
// relaxed remote arrive (no data changes hands); "dS written" needs a
// cluster-scope release, which costs the thread that issues it over a
// thousand cycles, so the elementwise warps arrive on a local barrier and an
// otherwise idle thread of that CTA (warp 2) forwards each completed phase.
//
// TMEM per CTA: dQ [0, 256) (quarters of 64 columns), X1 [256, 320), X2 [320,
// 384).  Warps: 0 producer A, 1 TMEM owner + MMA issuer A (first CTA of the
// pair), 2 MMA issuer B, 3 producer B, 4-7 elementwise + epilogue (thread t =
// TMEM lane t: query row t mod 64, key half t / 64).
#include <type_traits>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kX1 = 256, kX2 = 320;
constexpr int kHalf = kChunkBytes / 2;      // 64 rows x 64 columns
constexpr int kDsBytes = 2 * kHalf;         // dS: 64 rows x 128 keys
constexpr float kLog2e = 1.4426950408889634f;

// D = 64 NC with NC = 5..8: ceil(NC / 2) dQ quarters.
__host__ __device__ constexpr int n_quarters(int nc) { return (nc + 1) / 2; }
__host__ __device__ constexpr int grad_cols(int nc) { return 64 * n_quarters(nc); }  // TMEM columns of dQ per lane

// Ring slots of threads A and B: two of 16 KB each next to Q and dO (up to 128 KB).
constexpr int kSlot = kChunkBytes;
constexpr int kSlotsA = 2, kSlotsB = 2;
__host__ __device__ constexpr int res_bytes(int nc) { return 2 * nc * kHalf; }
__host__ __device__ constexpr int ds_off(int nc) { return res_bytes(nc); }
__host__ __device__ constexpr int ring_off(int nc) { return ds_off(nc) + 2 * kDsBytes; }
__host__ __device__ constexpr int bar_off(int nc) { return ring_off(nc) + (kSlotsA + kSlotsB) * kSlot; }
__host__ __device__ constexpr int smem_bytes(int nc) { return bar_off(nc) + 512 + 1024; }

struct Bars {
  int full_a, empty_a, full_b, empty_b, res_full, x1_full, x2_full, x1_free, x2_free, p_ready, acc_ready, drain_a,
      drain_b, p_local, count;  // p_ready, acc_ready, p_local: one per dS buffer
};
__host__ __device__ constexpr Bars bar_layout() {
  return Bars{0, kSlotsA, 2 * kSlotsA, 2 * kSlotsA + kSlotsB, 2 * (kSlotsA + kSlotsB), 2 * (kSlotsA + kSlotsB) + 1,
              2 * (kSlotsA + kSlotsB) + 2, 2 * (kSlotsA + kSlotsB) + 3, 2 * (kSlotsA + kSlotsB) + 4,
              2 * (kSlotsA + kSlotsB) + 5, 2 * (kSlotsA + kSlotsB) + 7, 2 * (kSlotsA + kSlotsB) + 9,
              2 * (kSlotsA + kSlotsB) + 10, 2 * (kSlotsA + kSlotsB) + 11, 2 * (kSlotsA + kSlotsB) + 13};
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
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Geometry of one CTA of a pair: its query tile and the key tiles it sweeps.
struct Geo {
  int b, h, kvh;  // batch, query head, kv head
  int st;         // query tile (128 rows)
  int s_row0;     // this CTA's first query row
  int ncols;      // key tiles (the same for both CTAs of the pair)
  int rot;        // the key sweep starts here
};

__device__ __forceinline__ Geo make_geo(const BwdParams& p, int rank) {
  Geo g;
  g.b = blockIdx.z;
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  g.st = p.q_tiles - 1 - pair;  // heavy causal tiles first
  g.h = blockIdx.y;
  g.kvh = g.h / p.group;
  const int kv_end = p.causal ? min(p.Nkv, (g.st + 1) * kTileRows) : p.Nkv;
  g.ncols = (kv_end + kTileRows - 1) / kTileRows;
  g.s_row0 = g.st * kTileRows + 64 * rank;
  g.rot = g.ncols > 0 ? g.st % g.ncols : 0;
  return g;
}

// first key row of key tile c
__device__ __forceinline__ int column(const Geo& g, int c) {
  c += g.rot;
  if (c >= g.ncols) c -= g.ncols;
  return c * kTileRows;
}

template <int NC, bool BF16, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_qh,
                  const __grid_constant__ CUtensorMap map_kh, const __grid_constant__ CUtensorMap map_vh,
                  const __grid_constant__ CUtensorMap map_doh, const __grid_constant__ BwdParams p) {
  constexpr int SA = kSlotsA, SB = kSlotsB;
  constexpr int kHps = kSlot / kHalf;    // score-operand half-chunks per slot
  constexpr int kResBytes = NC * kHalf;  // one resident operand: 64 rows x D columns
  constexpr int kNQ = n_quarters(NC);
  constexpr int kGradCols = grad_cols(NC);
  constexpr bool kPadded = (NC & 1) != 0;  // dQ columns past D
  constexpr Bars bl = bar_layout();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + bar_off(NC));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t a1_sm = smem_u32(smem), a2_sm = a1_sm + kResBytes, ds_sm = a1_sm + ds_off(NC);
  const uint32_t ring_a = a1_sm + ring_off(NC), ring_b = ring_a + SA * kSlot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const Geo g = make_geo(p, static_cast<int>(rank));
  uint32_t* status = p.status;
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  // resident A1 = Q, A2 = dO (64-row halves); score operands B1 = K, B2 = V
  // (64-row halves); dQ operand B3 = K (128 rows, MN-major)
  const CUtensorMap* mA1 = &map_qh;
  const CUtensorMap* mA2 = &map_doh;
  const CUtensorMap* mB1 = &map_kh;
  const CUtensorMap* mB2 = &map_vh;
  const CUtensorMap* mB3 = &map_k;

  if (tid == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(bar(bl.full_a + i), 1);
      mbar_init(bar(bl.empty_a + i), 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(bar(bl.full_b + i), 1);
      mbar_init(bar(bl.empty_b + i), 1);
    }
    mbar_init(bar(bl.res_full), 1);
    mbar_init(bar(bl.x1_full), 1);
    mbar_init(bar(bl.x2_full), 1);
    mbar_init(bar(bl.x1_free), 8);  // four elementwise warps in each CTA
    mbar_init(bar(bl.x2_free), 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.p_ready + i), 5);  // this CTA's four elementwise warps + the peer's relay
      mbar_init(bar(bl.p_local + i), 4);  // (second CTA) its four elementwise warps
      mbar_init(bar(bl.acc_ready + i), 2);  // gradient commits of threads A and B
    }
    mbar_init(bar(bl.drain_a), 1);
    mbar_init(bar(bl.drain_b), 1);
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
    // ------------------------------------------------------------ TMA producers (A: warp 0, B: warp 3)
    // Loads follow the order in which the ring's MMA thread uses them: the
    // score product of column 0; then, for each column c, the score product
    // of column c + 1 and the gradient quarters of column c.  The bytes of
    // both CTAs' loads are counted on the first CTA's full barrier.
    const bool is_a = warp == 0;
    const int S = is_a ? SA : SB;
    const int full0 = is_a ? bl.full_a : bl.full_b, empty0 = is_a ? bl.empty_a : bl.empty_b;
    const uint32_t ring = is_a ? ring_a : ring_b;
    tma_prefetch_desc(mB3);
    tma_prefetch_desc(is_a ? mB1 : mB2);
    if (is_a) {
      tma_prefetch_desc(mA1);
      if (rank == 0) mbar_expect_tx(bar(bl.res_full), 2 * res_bytes(NC));
      for (int c = 0; c < NC; ++c) {
        tma_load_4d_pair(a1_sm + c * kHalf, mA1, lead(bl.res_full), c * kChunk, g.s_row0, g.h, g.b);
        tma_load_4d_pair(a2_sm + c * kHalf, mA2, lead(bl.res_full), c * kChunk, g.s_row0, g.h, g.b);
      }
    }
    // Score product: half-chunks [x0, x1) of B1 or B2, kHps per slot (the
    // last slot may hold fewer).  dQ: quarters [q0, q1), one slot each holding
    // chunk 2 q + rank of B3.
    const CUtensorMap* mX = is_a ? mB1 : mB2;
    const int x0 = 0, x1 = NC;
    const int q0 = is_a ? 0 : 2, q1 = is_a ? 2 : kNQ;
    bool ok = true;
    uint32_t it = 0;
    auto next_slot = [&](uint32_t* dst, uint32_t* fb, int bytes) -> bool {
      const uint32_t s = it % S, r = it / S;
      ++it;
      if (!mbar_wait(bar(empty0 + s), (r & 1) ^ 1, status)) return false;
      *dst = ring + s * kSlot;
      *fb = lead(full0 + s);
      if (rank == 0) mbar_expect_tx(bar(full0 + s), 2 * bytes);
      return true;
    };
    auto x_loads = [&](int c) {
      const int ch = g.kvh, cr0 = column(g, c);
      for (int x = x0; x < x1 && ok; x += kHps) {
        const int n = min(kHps, x1 - x);
        uint32_t dst, fb;
        if (!(ok = next_slot(&dst, &fb, n * kHalf))) break;
        for (int i = 0; i < n; ++i)
          tma_load_4d_pair(dst + i * kHalf, mX, fb, (x + i) * kChunk, cr0 + 64 * static_cast<int>(rank), ch, g.b);
      }
    };
    auto g_loads = [&](int c) {
      const int ch = g.kvh, cr0 = column(g, c);
      for (int qd = q0; qd < q1 && ok; ++qd) {
        uint32_t dst, fb;
        if (!(ok = next_slot(&dst, &fb, kChunkBytes))) break;
        tma_load_4d_pair(dst, mB3, fb, (2 * qd + static_cast<int>(rank)) * kChunk, cr0, ch, g.b);
      }
    };
    if (g.ncols > 0) x_loads(0);
    for (int c = 0; c < g.ncols && ok; ++c) {
      if (c + 1 < g.ncols) x_loads(c + 1);
      g_loads(c);
    }
    // the ring's last commits (they arrive on both CTAs) complete before exit
    for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / S) * S;
      mbar_wait(bar(empty0 + s), (last / S) & 1, status);
    }
  } else if ((warp == 1 || warp == 2) && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuers A (warp 1) and B (warp 2)
    const bool is_a = warp == 1;
    const int S = is_a ? SA : SB;
    const int full0 = is_a ? bl.full_a : bl.full_b, empty0 = is_a ? bl.empty_a : bl.empty_b;
    const uint32_t ring = is_a ? ring_a : ring_b;
    const int xfull = is_a ? bl.x1_full : bl.x2_full, xfree = is_a ? bl.x1_free : bl.x2_free;
    const uint32_t x_tm = tbase + (is_a ? kX1 : kX2);
    constexpr uint32_t idesc_x = idesc_f16(BF16, 128, 128, false, false);  // 128 query rows x 128 keys
    constexpr uint32_t idesc_g = idesc_f16(BF16, 128, 128, false, true);   // 128 query rows x 128 dQ columns
    // resident operand of this thread's product: Q (S) or dO (dP)
    const uint64_t dres = sdesc_sw128(is_a ? a1_sm : a2_sm, 16, 1024);
    const uint64_t dring_k = sdesc_sw128(ring, 16, 1024);     // score operand: K-major half-chunks
    const uint64_t dring_m = sdesc_sw128(ring, kChunkBytes, 1024);  // dQ operand K: MN-major 64-column atoms
    const uint64_t dds = sdesc_sw128(ds_sm, 16, 1024);
    const int x0 = 0, x1 = NC;  // chunks of D this thread's product reduces over
    const int q0 = is_a ? 0 : 2;
    bool ok = mbar_wait(bar(bl.res_full), 0, status);
    tc_fence_after();
    uint32_t it = 0;
    auto wait_slot = [&]() -> uint32_t {
      const uint32_t s = it % S;
      ok = mbar_wait(bar(full0 + s), (it / S) & 1, status);
      ++it;
      tc_fence_after();
      return s;
    };
    // X (+)= A B^T over this thread's chunks of D, kHps chunks per slot
    auto product = [&]() {
      // Straight-line MMAs per slot where every slot is full: a bound check
      // between the MMAs of the issue loop slowed the kernels by 5%.
      constexpr int kSlotsX = (NC + 1) / 2;      // slots per product
      constexpr bool kRagged = (NC & 1) != 0;  // a slot with fewer than kHps chunks
      for (int m = 0; m < kSlotsX && ok; ++m) {
        const uint32_t s = wait_slot();
        if (!ok) return;
        const uint64_t bs = sdesc_advance(dring_k, s * kSlot);
#pragma unroll
        for (int i = 0; i < kHps; ++i) {
          if (kRagged && x0 + kHps * m + i >= x1) break;
          const uint64_t a = sdesc_advance(dres, (x0 + kHps * m + i) * kHalf);
          const uint64_t bd = sdesc_advance(bs, i * kHalf);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss_pair(x_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x, (m | i | kk) != 0);
        }
        umma_commit_pair(bar(empty0 + s), 3);
      }
    };
    // gradient += dS B3: A = dS (K-major, 128 column rows in two 64-row
    // subtiles), B = this CTA's 64 columns of the quarter (MN-major); quarters
    // [q0, q0 + nq)
    auto grad = [&](int c) {
      const uint64_t da = sdesc_advance(dds, (c & 1) * kDsBytes);
      const int nq = is_a ? 2 : kNQ - 2;  // dQ slots of this thread
      for (int qd = q0; qd < q0 + nq && ok; ++qd) {
        const uint32_t s = wait_slot();
        if (!ok) return;
        const uint64_t bs = sdesc_advance(dring_m, s * kSlot);
        const uint32_t acc_tm = tbase + 64 * qd;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_ss_pair(acc_tm, sdesc_advance(da, (ks >> 2) * kHalf + (ks & 3) * 32), sdesc_advance(bs, ks * 2048),
                       idesc_g, (c > 0 || ks > 0) ? 1u : 0u);
        umma_commit_pair(bar(empty0 + s), 3);
      }
    };
    if (g.ncols > 0 && ok) {
      product();
      if (ok) umma_commit_pair(bar(xfull), 3);
    }
    for (int c = 0; c < g.ncols && ok; ++c) {
      if (c + 1 < g.ncols) {
        // the elementwise warps have copied this column's scores (or dP) out of X
        ok = mbar_wait(bar(xfree), c & 1, status);
        if (!ok) break;
        tc_fence_after();
        product();
        if (!ok) break;
        umma_commit_pair(bar(xfull), 3);
      }
      ok = mbar_wait(bar(bl.p_ready + (c & 1)), (c >> 1) & 1, status);
      if (!ok) break;
      tc_fence_after();
      grad(c);
      if (!ok) break;
      umma_commit_pair(bar(bl.acc_ready + (c & 1)), 3);
    }
    const int drain = is_a ? bl.drain_a : bl.drain_b;
    umma_commit_pair(bar(drain), 1);
    mbar_wait(bar(drain), 0, status);
  } else if (warp == 2 && lane == 0 && rank == 1) {
    // ------------------------------------------------------------ relay of this CTA's p_ready
    // The elementwise warps of column c + 2 wait for the gradient MMAs of
    // column c, which need this relay's arrive: p_local cannot run two phases
    // ahead of this loop.
    for (int c = 0; c < g.ncols; ++c) {
      if (!mbar_wait(bar(bl.p_local + (c & 1)), (c >> 1) & 1, status)) break;
      mbar_arrive_remote(lead(bl.p_ready + (c & 1)));  // release.cluster: the dS tile is visible first
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise + epilogue
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int t = tid - 128;  // TMEM lane
    const int r = t & 63;     // query row within this CTA's 64
    const int u = t >> 6;     // key half of the key tile
    const int srow = g.s_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t x1_free_lead = lead(bl.x1_free), x2_free_lead = lead(bl.x2_free);
    const uint32_t p_ready0 = bar(rank == 0 ? bl.p_ready : bl.p_local);  // local: the first CTA's or the relay's
    float lse2_row, delta_row;
    {
      const int64_t idx = (static_cast<int64_t>(g.b) * p.Hq + g.h) * p.Nq + min(srow, p.Nq - 1);
      lse2_row = p.lse2[idx];
      delta_row = p.delta[idx];
    }
    const DropKey dkey = {p.drop_seed_lo, p.drop_seed_hi, static_cast<uint32_t>(g.b * p.Hq + g.h), p.drop_off,
                          p.drop_t};
    bool ok = true;
    auto arrive_free = [&](uint32_t a) {  // "X consumed": no data hand-off
      if (rank == 0)
        mbar_arrive(a);
      else
        mbar_arrive_remote_relaxed(a);
    };
    auto load64 = [&](uint32_t col, float (&f)[64]) {
      uint32_t a0[32], a1[32];
      tmem_ld32(tbase + lane_off + col, a0);
      tmem_ld32(tbase + lane_off + col + 32, a1);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        f[e] = __uint_as_float(a0[e]);
        f[32 + e] = __uint_as_float(a1[e]);
      }
    };
    for (int c = 0; c < g.ncols; ++c) {
      const int cbase = column(g, c) + 64 * u;  // first key of this thread's half
      bool plain = srow < p.Nq && cbase + 64 <= p.Nkv && (!p.causal || cbase + 63 <= srow) && lse2_row > -INFINITY;
      plain = __all_sync(0xffffffffu, plain) && p.bias == nullptr;
      // dropout: the keep bits of this thread's 64 keys, drawn while S is computed
      uint32_t keep_lo = 0, keep_hi = 0;
      if constexpr (DROP) keep64_row(dkey, cbase, srow, keep_lo, keep_hi);

      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x1_full), c & 1, status));
      if (!ok) break;
      float pv[64];
      tc_fence_after();
      load64(kX1, pv);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_free(x1_free_lead);
      // P = 2^(S scale log2e + bias log2e - lse2), 0 where masked
      if (plain) {
#pragma unroll
        for (int e = 0; e < 64; ++e) pv[e] = ex2(fmaf(pv[e], p.scale_log2, -lse2_row));
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int i = srow, j = cbase + e;
          const bool valid = i < p.Nq && j < p.Nkv && !(p.causal && j > i) && lse2_row > -INFINITY;
          float xv = fmaf(pv[e], p.scale_log2, -lse2_row);
          if (p.bias)
            xv = fmaf(__ldg(p.bias + g.b * p.bias_sb + g.h * p.bias_sh +
                            static_cast<int64_t>(min(i, p.Nq - 1)) * p.bias_sq +
                            static_cast<int64_t>(min(j, p.Nkv - 1)) * p.bias_sk),
                      kLog2e, xv);
          pv[e] = valid ? ex2(xv) : 0.f;
        }
      }
      {
        // dS = P (dP - Delta)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x2_full), c & 1, status));
        if (!ok) break;
        tc_fence_after();
        float dp[64];
        load64(kX2, dp);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_free(x2_free_lead);
        if constexpr (DROP) {
          // dP of the dropped output: dO V^T times keep / (1 - p)
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const bool kept = (((e < 32 ? keep_lo : keep_hi) >> (e & 31)) & 1u) != 0;
            pv[e] *= (kept ? dp[e] * p.drop_scale : 0.f) - delta_row;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) pv[e] *= dp[e] - delta_row;
        }
      }
      uint32_t w[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) w[e] = pack2<BF16>(pv[2 * e], pv[2 * e + 1]);
      if (c >= 2) {
        // the gradient MMAs of column c - 2 read this dS buffer.  Those of
        // column c cannot have completed yet, so the parity is unambiguous.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready + (c & 1)), ((c - 2) >> 1) & 1, status));
        if (!ok) break;
      }
      {
        // row r of the K-major, 128-byte-swizzled [64 rows x 64 columns] subtile u
        const uint32_t row = ds_sm + static_cast<uint32_t>(c & 1) * kDsBytes + static_cast<uint32_t>(u) * kHalf +
                             static_cast<uint32_t>(r) * 128u;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_shared_v4(row + ((static_cast<uint32_t>(q) ^ static_cast<uint32_t>(r & 7)) << 4), w[4 * q],
                       w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready0 + 8 * (c & 1));
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      // the last dQ MMAs of each dS buffer (their commits also arrive on the peer)
      if (g.ncols > 0)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(bl.acc_ready + ((g.ncols - 1) & 1)), ((g.ncols - 1) >> 1) & 1, status));
      if (ok && g.ncols > 1)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready + (g.ncols & 1)), ((g.ncols - 2) >> 1) & 1, status));
      if (ok && g.ncols > 0) tc_fence_after();
      if (ok) {
        T* dst_base = reinterpret_cast<T*>(p.dq);
        const int64_t sb = p.dq_sb, sh = p.dq_sh, sn = p.dq_sn;
        const float mul = p.scale;
        T* orow = dst_base + g.b * sb + g.h * sh + static_cast<int64_t>(srow) * sn;
        for (int k = 0; k < kGradCols / 32; ++k) {
          // TMEM column 64 qd + 32 hh + e of lane 64 u + r is D column 128 qd +
          // 64 u + 32 hh + e
          const int tcol = 32 * k;
          const int dcol = 128 * (k >> 1) + 64 * u + 32 * (k & 1);
          if (kPadded && dcol >= 64 * NC) continue;  // zero-filled operand columns past D
          {
            uint32_t v[32];
            if (g.ncols > 0) {
              tmem_ld32(tbase + lane_off + tcol, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (srow < p.Nq) {
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
cudaError_t launch_impl(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  constexpr int smem = smem_bytes(NC);
  static_assert(smem <= 232448, "shared memory per CTA");
  static_assert(grad_cols(NC) <= 256, "dQ below the score buffers");
  auto kern = p.dropout ? bwd_dq_kernel<NC, BF16, true> : bwd_dq_kernel<NC, BF16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.q_tiles, p.Hq, p.B);
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
  e = cudaLaunchKernelEx(&cfg, kern, m.k, m.q_half, m.k_half, m.v_half, m.dout_half, p);
  timing_mark(st);
  return e;
}

template <bool BF16>
cudaError_t launch_dq(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  switch (p.n_chunks) {
    case 5: return launch_impl<5, BF16>(p, m, st);
    case 6: return launch_impl<6, BF16>(p, m, st);
    case 7: return launch_impl<7, BF16>(p, m, st);
    default: return launch_impl<8, BF16>(p, m, st);
  }
}

}  // namespace

bool bwd_dq_supported(const BwdParams& p) { return p.n_chunks >= 5 && p.n_chunks <= 8; }

cudaError_t launch_bwd_dq(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_dq<true>(p, m, s) : launch_dq<false>(p, m, s);
}

}  // namespace ffpa
