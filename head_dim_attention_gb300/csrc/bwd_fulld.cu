// Attention backward for D = 512: dV, dK and dQ kernels in which a CTA pair
// holds ALL of D (tcgen05 cta_group::2 with M = 128).  Same decomposition as
// bwd.cu (FFPA Attention Benchmark page, "More Benchmark": preprocess, dV, dK,
// dQ, 8 GEMM passes): P is rebuilt from the forward's lse, and
//   dV:  S^T = K Q^T,  P^T,                      dV += P^T dO      (2 GEMMs)
//   dK:  S^T, dP^T = V dO^T, dS^T = P^T (dP^T - Delta),  dK += dS^T Q (3 GEMMs)
//   dQ:  S = Q K^T, dP = dO V^T, dS = P (dP - Delta),     dQ += dS K  (3 GEMMs)
//
// Why M = 128 pairs.  A 128 x 512 fp32 gradient fills a CTA's 512 TMEM
// columns, so a one-CTA kernel (or an M = 256 pair) must split the gradient's
// columns over CTAs that each recompute the score products over the whole of
// D.  With cta_group::2 and M = 128 each SM holds 64 rows of the accumulator
// across all 128 TMEM lanes (lane r: row r, the first N/2 columns; lane r + 64:
// row r, the other N/2), so the 128 x 512 gradient of a stationary tile takes
// 256 columns per SM and the score products are computed once: 16 Nq Nkv D
// executed per head instead of 26.
//
// Per pair: one 128-row stationary tile (key rows for dV/dK, query rows for
// dQ); CTA c of the pair holds rows 64c .. 64c + 63 of it and keeps its
// stationary operands resident in shared memory (K for dV; K and V for dK; Q
// and dO for dQ), 64 rows x 512 columns each.  The kernel sweeps 128-row column
// tiles (query tiles of every query head of the GQA group for dV/dK, key tiles
// for dQ).  Per column tile:
//   X1 = scores    M=128, N=128 (B split by N: CTA c loads column rows 64c..),
//                  reduced over the eight 64-column chunks of D
//   X2 = dP        the same with the second stationary operand (dK, dQ)
//   dS (or P)      elementwise, rounded to the input type, written to shared
//                  memory as the K-major A operand (64 rows x 128 columns), in
//                  two buffers used by alternate column tiles, so the
//                  elementwise warps write one while the gradient MMAs read
//                  the other
//   gradient       dK, dQ: four quarters of D, M=128, N=128: CTA c supplies
//                  the 64 columns 128 qd + 64 c .. of the column operand
//                  (MN-major); dV: two halves of D, M=128, N=256: CTA c
//                  supplies the 128 columns 256 h + 128 c ..
// Each of these pair MMAs costs the issuing thread more time than the tensor
// core needs for it, and each barrier wait costs it about as much as four
// MMAs, so one thread cannot keep the tensor core busy.  Two threads issue:
//   thread A: X1 and gradient quarters 0, 1;  thread B: X2 and quarters 2, 3
// (dV: thread A reduces X1 over chunks 0..3 and thread B over chunks 4..7 into
// two accumulators that the elementwise warps add, and each accumulates one
// half of dV).  Each issuing thread has its own ring with its own TMA
// producer, so every ring keeps a single producer and a single consumer.
// dK and dQ keep two stationary operands resident and fit four 16 KB slots;
// dV keeps one and uses four 32 KB slots (fewer, larger barrier phases: each
// of its threads waits twice per column tile instead of four times).
//
// Signals from the second CTA of the pair to the first: "X consumed" is a
// relaxed remote arrive (no data changes hands); "dS written" needs a
// cluster-scope release, which costs the thread that issues it over a
// thousand cycles, so the elementwise warps arrive on a local barrier and an
// otherwise idle thread of that CTA (warp 2) forwards each completed phase.
//
// TMEM per CTA: gradient [0, 256) (dK, dQ: quarters of 64 columns; dV: halves
// of 128), X1 [256, 320), X2 [320, 384).  Warps: 0 producer A, 1 TMEM owner + MMA issuer A (first CTA
// of the pair), 2 MMA issuer B, 3 producer B, 4-7 elementwise + epilogue
// (thread t = TMEM lane t: stationary row t mod 64, column half t / 64).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

enum Mode : int { kDV = 0, kDK = 1, kDQ = 2 };

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kX1 = 256, kX2 = 320;
constexpr int kHalf = kChunkBytes / 2;      // 64 rows x 64 columns
constexpr int kDsBytes = 2 * kHalf;         // dS or P: 64 rows x 128 columns
constexpr float kLog2e = 1.4426950408889634f;

// D = 64 NC with NC = 5..8.  The score products reduce over the NC chunks.
// The gradient runs in quarters of 128 columns (dK, dQ; ceil(NC / 2) of them)
// or in two halves (dV: columns 0..255 and 256 .. 256 + N1 - 1, N1 = 256 for
// D > 384, else 128); gradient operand columns at or past D are zero-filled
// by TMA and the matching gradient columns are not stored.
__host__ __device__ constexpr int n_quarters(int nc) { return (nc + 1) / 2; }
__host__ __device__ constexpr int dv_n1(int nc) { return nc >= 7 ? 256 : 128; }
// TMEM columns of the gradient per lane
__host__ __device__ constexpr int grad_cols(int mode, int nc) { return mode == kDV ? 128 + dv_n1(nc) / 2 : 64 * n_quarters(nc); }

// Ring slots of threads A and B: dK and dQ keep two operands resident (up to
// 128 KB) and use two 16 KB slots each; dV keeps one and uses two of 32 KB.
__host__ __device__ constexpr int slot_bytes(int mode) { return mode == kDV ? 2 * kChunkBytes : kChunkBytes; }
__host__ __device__ constexpr int slots_a(int mode) { return 2; }
__host__ __device__ constexpr int slots_b(int mode) { return 2; }
__host__ __device__ constexpr int res_bytes(int mode, int nc) { return (mode == kDV ? 1 : 2) * nc * kHalf; }
__host__ __device__ constexpr int ds_off(int mode, int nc) { return res_bytes(mode, nc); }
__host__ __device__ constexpr int ring_off(int mode, int nc) { return ds_off(mode, nc) + 2 * kDsBytes; }
__host__ __device__ constexpr int bar_off(int mode, int nc) {
  return ring_off(mode, nc) + (slots_a(mode) + slots_b(mode)) * slot_bytes(mode);
}
__host__ __device__ constexpr int smem_bytes(int mode, int nc) { return bar_off(mode, nc) + 512 + 1024; }

struct Bars {
  int full_a, empty_a, full_b, empty_b, res_full, x1_full, x2_full, x1_free, x2_free, p_ready, acc_ready, drain_a,
      drain_b, p_local, count;  // p_ready, acc_ready, p_local: one per dS buffer
};
__host__ __device__ constexpr Bars bar_layout(int mode) {
  return Bars{0,
              slots_a(mode),
              2 * slots_a(mode),
              2 * slots_a(mode) + slots_b(mode),
              2 * (slots_a(mode) + slots_b(mode)),
              2 * (slots_a(mode) + slots_b(mode)) + 1,
              2 * (slots_a(mode) + slots_b(mode)) + 2,
              2 * (slots_a(mode) + slots_b(mode)) + 3,
              2 * (slots_a(mode) + slots_b(mode)) + 4,
              2 * (slots_a(mode) + slots_b(mode)) + 5,
              2 * (slots_a(mode) + slots_b(mode)) + 7,
              2 * (slots_a(mode) + slots_b(mode)) + 9,
              2 * (slots_a(mode) + slots_b(mode)) + 10,
              2 * (slots_a(mode) + slots_b(mode)) + 11,
              2 * (slots_a(mode) + slots_b(mode)) + 13};
}
static_assert(bar_layout(kDV).count * 8 + 16 <= 512, "barrier area");

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

// Stationary/column geometry of one CTA of a pair.
struct Geo {
  int b, h, kvh;       // batch, query head (dQ) and kv head
  int st;              // stationary tile (128 rows)
  int s_head, s_row0;  // this CTA's 64 stationary rows: head index in its tensor, first row
  int s_limit;         // rows of the stationary tensor
  int qt_begin, nq_h;  // dV/dK: first query tile and query tiles per head
  int ncols;           // column tiles (the same for both CTAs of the pair)
  int rot;             // the column sweep starts here
};

template <int MODE>
__device__ __forceinline__ Geo make_geo(const BwdParams& p, int rank) {
  Geo g;
  g.b = blockIdx.z;
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  if (MODE == kDQ) {
    g.st = p.q_tiles - 1 - pair;  // heavy causal tiles first
    g.h = blockIdx.y;
    g.kvh = g.h / p.group;
    g.s_head = g.h;
    g.s_limit = p.Nq;
    const int kv_end = p.causal ? min(p.Nkv, (g.st + 1) * kTileRows) : p.Nkv;
    g.ncols = (kv_end + kTileRows - 1) / kTileRows;
    g.qt_begin = 0;
    g.nq_h = 0;
  } else {
    g.st = pair;
    g.kvh = blockIdx.y;
    g.h = g.kvh * p.group;
    g.s_head = g.kvh;
    g.s_limit = p.Nkv;
    g.qt_begin = p.causal ? g.st : 0;  // top-left causal: query rows i >= key row j
    g.nq_h = max(0, p.q_tiles - g.qt_begin);
    g.ncols = p.group * g.nq_h;
  }
  g.s_row0 = g.st * kTileRows + 64 * rank;
  g.rot = g.ncols > 0 ? g.st % g.ncols : 0;
  return g;
}

template <int MODE>
__device__ __forceinline__ void column(const Geo& g, const BwdParams& p, int c, int* head, int* row0) {
  c += g.rot;
  if (c >= g.ncols) c -= g.ncols;
  if (MODE == kDQ) {
    *head = g.kvh;
    *row0 = c * kTileRows;
  } else {
    *head = g.kvh * p.group + c / g.nq_h;
    *row0 = (g.qt_begin + c % g.nq_h) * kTileRows;
  }
}

template <int MODE, int NC, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_fulld_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                     const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                     const __grid_constant__ CUtensorMap map_vh, const __grid_constant__ CUtensorMap map_doh,
                     const __grid_constant__ BwdParams p) {
  constexpr bool TWO = MODE != kDV;  // a dP product (X2); dV splits X1 over two accumulators instead
  constexpr int SA = slots_a(MODE), SB = slots_b(MODE);
  constexpr int kSlot = slot_bytes(MODE);
  constexpr int kHps = kSlot / kHalf;                  // score-operand half-chunks per slot
  constexpr int kResBytes = NC * kHalf;                // one stationary operand: 64 rows x D columns
  constexpr int kNQ = n_quarters(NC), kN1 = dv_n1(NC);
  constexpr int kGradCols = grad_cols(MODE, NC);
  constexpr bool kPadded = TWO ? (NC & 1) != 0 : 64 * NC < 256 + kN1;  // gradient columns past D
  constexpr Bars bl = bar_layout(MODE);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + bar_off(MODE, NC));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t a1_sm = smem_u32(smem), a2_sm = a1_sm + kResBytes, ds_sm = a1_sm + ds_off(MODE, NC);
  const uint32_t ring_a = a1_sm + ring_off(MODE, NC), ring_b = ring_a + SA * kSlot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const Geo g = make_geo<MODE>(p, static_cast<int>(rank));
  uint32_t* status = p.status;
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  // stationary A1, A2 (64-row halves); column operands B1, B2 (64-row halves); gradient operand B3 (128 rows)
  const CUtensorMap* mA1 = (MODE == kDQ) ? &map_qh : &map_kh;
  const CUtensorMap* mA2 = (MODE == kDQ) ? &map_doh : &map_vh;
  const CUtensorMap* mB1 = (MODE == kDQ) ? &map_kh : &map_qh;
  const CUtensorMap* mB2 = (MODE == kDQ) ? &map_vh : &map_doh;
  const CUtensorMap* mB3 = (MODE == kDV) ? &map_do : ((MODE == kDK) ? &map_q : &map_k);

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
    tma_prefetch_desc(is_a ? mB1 : (TWO ? mB2 : mB1));
    if (is_a) {
      tma_prefetch_desc(mA1);
      if (rank == 0) mbar_expect_tx(bar(bl.res_full), 2 * res_bytes(MODE, NC));
      for (int c = 0; c < NC; ++c) {
        tma_load_4d_pair(a1_sm + c * kHalf, mA1, lead(bl.res_full), c * kChunk, g.s_row0, g.s_head, g.b);
        if (TWO) tma_load_4d_pair(a2_sm + c * kHalf, mA2, lead(bl.res_full), c * kChunk, g.s_row0, g.s_head, g.b);
      }
    }
    // Score product: half-chunks [x0, x1) of B1 or B2, kHps per slot (the
    // last slot may hold fewer).  Gradient: dK, dQ: quarters [q0, q1), one slot
    // each holding chunk 2 q + rank of B3; dV: half h, one slot holding this
    // CTA's one or two chunks of it.
    const CUtensorMap* mX = (is_a || !TWO) ? mB1 : mB2;
    const int x0 = (!TWO && !is_a) ? 4 : 0, x1 = (!TWO && is_a) ? 4 : NC;
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
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      for (int x = x0; x < x1 && ok; x += kHps) {
        const int n = min(kHps, x1 - x);
        uint32_t dst, fb;
        if (!(ok = next_slot(&dst, &fb, n * kHalf))) break;
        for (int i = 0; i < n; ++i)
          tma_load_4d_pair(dst + i * kHalf, mX, fb, (x + i) * kChunk, cr0 + 64 * static_cast<int>(rank), ch, g.b);
      }
    };
    auto g_loads = [&](int c) {
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      if constexpr (TWO) {
        for (int qd = q0; qd < q1 && ok; ++qd) {
          uint32_t dst, fb;
          if (!(ok = next_slot(&dst, &fb, kChunkBytes))) break;
          tma_load_4d_pair(dst, mB3, fb, (2 * qd + static_cast<int>(rank)) * kChunk, cr0, ch, g.b);
        }
      } else {
        const int hf = is_a ? 0 : 1, nv = (hf == 0 || kN1 == 256) ? 2 : 1;
        uint32_t dst, fb;
        if (!(ok = next_slot(&dst, &fb, nv * kChunkBytes))) return;
        for (int i = 0; i < nv; ++i)
          tma_load_4d_pair(dst + i * kChunkBytes, mB3, fb, (4 * hf + nv * static_cast<int>(rank) + i) * kChunk, cr0,
                           ch, g.b);
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
    constexpr uint32_t idesc_x = idesc_f16(BF16, 128, 128, false, false);  // 128 stationary rows x 128 columns
    // stationary rows x gradient columns (dV: half 0, then half 1 of N1 columns)
    constexpr uint32_t idesc_g = idesc_f16(BF16, 128, TWO ? 128 : 256, false, true);
    constexpr uint32_t idesc_g1 = idesc_f16(BF16, 128, TWO ? 128 : kN1, false, true);
    // resident stationary operand of this thread's product (dV: K for both halves of D)
    const uint64_t dres = sdesc_sw128((is_a || !TWO) ? a1_sm : a2_sm, 16, 1024);
    const uint64_t dring_k = sdesc_sw128(ring, 16, 1024);     // score operand: K-major half-chunks
    const uint64_t dring_m = sdesc_sw128(ring, kChunkBytes, 1024);  // gradient operand: MN-major 64-column atoms 16 KB apart
    const uint64_t dds = sdesc_sw128(ds_sm, 16, 1024);
    const int x0 = (!TWO && !is_a) ? 4 : 0, x1 = (!TWO && is_a) ? 4 : NC;
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
      constexpr int kSlotsX = TWO ? (NC + 1) / 2 : 1;       // slots per product (dV: 4 or NC - 4 chunks)
      constexpr bool kRagged = TWO ? (NC & 1) != 0 : NC != 8;  // a slot with fewer than kHps chunks
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
    // subtiles), B = this CTA's columns of the quarter (64) or half (128) of D
    // (MN-major); dK, dQ: quarters [q0, q1), dV: half q0 / 2
    auto grad = [&](int c) {
      const uint64_t da = sdesc_advance(dds, (c & 1) * kDsBytes);
      constexpr bool kSameG = idesc_g == idesc_g1;
      const uint32_t idg = (kSameG || TWO || is_a) ? idesc_g : idesc_g1;
      const int nq = TWO ? (is_a ? 2 : kNQ - 2) : 1;  // gradient slots of this thread
      for (int qd = q0; qd < q0 + nq && ok; ++qd) {
        const uint32_t s = wait_slot();
        if (!ok) return;
        const uint64_t bs = sdesc_advance(dring_m, s * kSlot);
        const uint32_t acc_tm = tbase + (TWO ? 64 * qd : 64 * q0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_ss_pair(acc_tm, sdesc_advance(da, (ks >> 2) * kHalf + (ks & 3) * 32), sdesc_advance(bs, ks * 2048),
                       idg, (c > 0 || ks > 0) ? 1u : 0u);
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
    const int r = t & 63;     // stationary row within this CTA's 64
    const int u = t >> 6;     // column half of the column tile
    const int srow = g.s_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t x1_free_lead = lead(bl.x1_free), x2_free_lead = lead(bl.x2_free);
    const uint32_t p_ready0 = bar(rank == 0 ? bl.p_ready : bl.p_local);  // local: the first CTA's or the relay's
    float lse2_row = 0.f, delta_row = 0.f;
    if (MODE == kDQ) {
      const int64_t idx = (static_cast<int64_t>(g.b) * p.Hq + g.h) * p.Nq + min(srow, p.Nq - 1);
      lse2_row = p.lse2[idx];
      delta_row = p.delta[idx];
    }
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
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      const int cbase = cr0 + 64 * u;  // first column row of this thread's half
      // Column statistics (dV, dK): lane l holds lse2 and Delta of column rows
      // cbase + l and cbase + 32 + l; threads take theirs with shuffles.
      float l2v[2] = {0.f, 0.f}, dlv[2] = {0.f, 0.f};
      if (MODE != kDQ) {
        const int64_t sbase = (static_cast<int64_t>(g.b) * p.Hq + ch) * p.Nq;
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int64_t i = sbase + min(cbase + 32 * k2 + lane, p.Nq - 1);
          l2v[k2] = p.lse2[i];
          if (TWO) dlv[k2] = p.delta[i];
        }
      }
      bool plain;
      if (MODE == kDQ)
        plain = srow < p.Nq && cbase + 64 <= p.Nkv && (!p.causal || cbase + 63 <= srow) && lse2_row > -INFINITY;
      else
        plain = srow < p.Nkv && cbase + 64 <= p.Nq && (!p.causal || srow <= cbase);
      plain = __all_sync(0xffffffffu, plain) && p.bias == nullptr;

      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x1_full), c & 1, status));
      if (!ok) break;
      float pv[64];
      if constexpr (!TWO) {
        // dV: the two halves of D were reduced into X1 and X2
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x2_full), c & 1, status));
        if (!ok) break;
        tc_fence_after();
        float q[64];
        load64(kX1, pv);
        load64(kX2, q);
#pragma unroll
        for (int e = 0; e < 64; ++e) pv[e] += q[e];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          arrive_free(x1_free_lead);
          arrive_free(x2_free_lead);
        }
      } else {
        tc_fence_after();
        load64(kX1, pv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_free(x1_free_lead);
      }
      // P = 2^(S scale log2e + bias log2e - lse2), 0 where masked
      if (plain) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float l2 = (MODE == kDQ) ? lse2_row : __shfl_sync(0xffffffffu, l2v[e >> 5], e & 31);
          pv[e] = ex2(fmaf(pv[e], p.scale_log2, -l2));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          int i, j;
          float l2;
          if (MODE == kDQ) {
            i = srow;
            j = cbase + e;
            l2 = lse2_row;
          } else {
            i = cbase + e;
            j = srow;
            l2 = __shfl_sync(0xffffffffu, l2v[e >> 5], e & 31);
          }
          const int hq = (MODE == kDQ) ? g.h : ch;
          const bool valid = i < p.Nq && j < p.Nkv && !(p.causal && j > i) && l2 > -INFINITY;
          float xv = fmaf(pv[e], p.scale_log2, -l2);
          if (p.bias)
            xv = fmaf(__ldg(p.bias + g.b * p.bias_sb + hq * p.bias_sh +
                            static_cast<int64_t>(min(i, p.Nq - 1)) * p.bias_sq +
                            static_cast<int64_t>(min(j, p.Nkv - 1)) * p.bias_sk),
                      kLog2e, xv);
          pv[e] = valid ? ex2(xv) : 0.f;
        }
      }
      if constexpr (TWO) {
        // dS = P (dP - Delta)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x2_full), c & 1, status));
        if (!ok) break;
        tc_fence_after();
        float dp[64];
        load64(kX2, dp);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_free(x2_free_lead);
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float dl = (MODE == kDQ) ? delta_row : __shfl_sync(0xffffffffu, dlv[e >> 5], e & 31);
          pv[e] *= dp[e] - dl;
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
      // the last gradient MMAs of each dS buffer (their commits also arrive on the peer)
      if (g.ncols > 0)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(bl.acc_ready + ((g.ncols - 1) & 1)), ((g.ncols - 1) >> 1) & 1, status));
      if (ok && g.ncols > 1)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready + (g.ncols & 1)), ((g.ncols - 2) >> 1) & 1, status));
      if (ok && g.ncols > 0) tc_fence_after();
      if (ok) {
        T* dst_base;
        int64_t sb, sh, sn;
        if (MODE == kDV) {
          dst_base = reinterpret_cast<T*>(p.dv); sb = p.dv_sb; sh = p.dv_sh; sn = p.dv_sn;
        } else if (MODE == kDK) {
          dst_base = reinterpret_cast<T*>(p.dk); sb = p.dk_sb; sh = p.dk_sh; sn = p.dk_sn;
        } else {
          dst_base = reinterpret_cast<T*>(p.dq); sb = p.dq_sb; sh = p.dq_sh; sn = p.dq_sn;
        }
        const float mul = (MODE == kDV) ? 1.f : p.scale;
        T* orow = dst_base + g.b * sb + g.s_head * sh + static_cast<int64_t>(srow) * sn;
        for (int k = 0; k < kGradCols / 32; ++k) {
          // dK, dQ: TMEM column 64 qd + 32 hh + e of lane 64 u + r is D column
          // 128 qd + 64 u + 32 hh + e; dV: column 128 h + 32 hh + e is D column
          // 256 h + (N_h / 2) u + 32 hh + e (N_0 = 256, N_1 = N1)
          const int tcol = 32 * k;
          const int dcol = TWO ? 128 * (k >> 1) + 64 * u + 32 * (k & 1)
                               : ((k < 4 || kN1 == 256) ? 256 * (k >> 2) + 128 * u + 32 * (k & 3)
                                                        : 256 + 64 * u + 32 * (k - 4));
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
            if (srow < g.s_limit) {
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

template <int MODE, int NC, bool BF16>
cudaError_t launch_mode(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  constexpr int smem = smem_bytes(MODE, NC);
  static_assert(smem <= 232448, "shared memory per CTA");
  static_assert(grad_cols(MODE, NC) <= 256, "gradient below the score buffers");
  auto kern = bwd_fulld_kernel<MODE, NC, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (MODE == kDQ) ? p.q_tiles : p.kv_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = (MODE == kDQ) ? dim3(2 * tiles, p.Hq, p.B) : dim3(2 * tiles, p.Hkv, p.B);
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
  e = cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, m.dout, m.q_half, m.k_half, m.v_half, m.dout_half, p);
  timing_mark(st);
  return e;
}

template <bool BF16>
cudaError_t launch_dq(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  switch (p.n_chunks) {
    case 5: return launch_mode<kDQ, 5, BF16>(p, m, st);
    case 6: return launch_mode<kDQ, 6, BF16>(p, m, st);
    case 7: return launch_mode<kDQ, 7, BF16>(p, m, st);
    default: return launch_mode<kDQ, 8, BF16>(p, m, st);
  }
}

}  // namespace

bool bwd_fulld_supported(const BwdParams& p) { return p.n_chunks >= 5 && p.n_chunks <= 8; }

cudaError_t launch_bwd_fulld_dq(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_dq<true>(p, m, s) : launch_dq<false>(p, m, s);
}

}  // namespace ffpa
