// Attention backward for D = 512, CTA-pair flavour of the dV, dK and dQ
// kernels of bwd.cu (same decomposition, from the FFPA Attention Benchmark
// page, "More Benchmark": preprocess, dV, dK, dQ, 8 GEMM passes).
//
// Each kernel keeps a 128-row tile stationary (key rows for dV/dK, query rows
// for dQ) and sweeps 128-row column tiles; the gradient's 512 columns are
// split in two halves of 256, and every CTA owning a half reduces the score
// products over the whole of D (TMEM cannot hold a 128 x 512 fp32 gradient
// next to the score tiles).  Here the two CTAs that own the SAME half for two
// neighbouring stationary tiles form a cluster and issue their MMAs as one
// pair (tcgen05 cta_group::2, M = 256):
//   * score products (X1 = S or S^T; X2 = dP or dP^T): each CTA supplies its
//     own stationary operand as A and HALF of the column tile (64 rows x 512)
//     as B, and receives its own 128 x 128 product;
//   * gradient (dV += P^T dO, dK += dS^T Q, dQ += dS K): each CTA supplies its
//     own P or dS from TMEM as A and HALF of the gradient half's columns of
//     the column operand (128 rows x 128) as B.
// Per column tile an SM loads the column tensor's bytes once between the
// pair instead of twice, and its shared memory serves half of each B operand.
//
// TMEM per CTA: gradient [0, 256), X1 [256, 384), X2 [384, 512).  Shared
// memory, dV: K resident (128 KB) and a ring of three 32 KB slots, each
// holding four 64-row column half-chunks or this CTA's two gradient-operand
// chunks.  dK and dQ need two stationary operands (K and V, or Q and dO) that
// do not both fit, and streaming one of them through a short ring left the
// second product waiting on loads; so both stream, through four 48 KB slots
// that each hold two 128-row stationary chunks next to the matching two
// column half-chunks (or the two gradient-operand chunks).
// Warp roles as in bwd.cu; the first CTA of the pair issues the MMAs.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

enum Mode : int { kDV = 0, kDK = 1, kDQ = 2 };

constexpr int kThreads = 256;
constexpr int kProducers = 3;  // warps 0, 2 and 3
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kX1 = 256, kX2 = 384;
constexpr int kChunks = 8;                       // D = 512
constexpr int kHalfChunkBytes = kChunkBytes / 2;  // 64 rows x 64 columns
// dV: resident K and 32 KB slots; dK/dQ: nothing resident and 48 KB slots
__host__ __device__ constexpr int res_bytes(int mode) { return mode == kDV ? kChunks * kChunkBytes : 0; }
__host__ __device__ constexpr int slot_bytes(int mode) { return mode == kDV ? 2 * kChunkBytes : 3 * kChunkBytes; }
constexpr float kLog2e = 1.4426950408889634f;

struct Bars {
  int full, empty, a_full, x1_full, x2_full, x1_free, p_ready, acc_ready, drain, count;
};
__host__ __device__ inline Bars bar_layout(int stages) {
  Bars b;
  b.full = 0;
  b.empty = stages;
  b.a_full = 2 * stages;
  b.x1_full = b.a_full + 1;
  b.x2_full = b.x1_full + 1;
  b.x1_free = b.x2_full + 1;
  b.p_ready = b.x1_free + 1;
  b.acc_ready = b.p_ready + 1;
  b.drain = b.acc_ready + 1;
  b.count = b.drain + 1;
  return b;
}
// dK: each elementwise warp stages its column tile's statistics (lse2 and
// Delta of 128 column rows, 1 KB) in shared memory
__host__ __device__ constexpr int stat_bytes(int mode) { return mode == kDK ? 4 * 1024 : 0; }
__host__ __device__ constexpr int smem_bytes(int mode, int stages) {
  return res_bytes(mode) + stages * slot_bytes(mode) + 1024 + stat_bytes(mode) + 1024;
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

// Stationary/column geometry of one CTA of a pair.
struct Geo {
  int b, h, kvh;       // batch, query head (dQ) and kv head
  int s_head, s_row0;  // stationary tile: head index in its tensor, first row
  int s_limit;         // rows of the stationary tensor
  int qt_begin, nq_h;  // dV/dK: first query tile and query tiles per head
  int ncols;           // column tiles (the same for both CTAs of the pair)
  int rot;             // the column sweep starts here
  int dh;              // half of D the pair's gradient covers
};

template <int MODE>
__device__ __forceinline__ Geo make_geo(const BwdParams& p, int rank) {
  Geo g;
  g.b = blockIdx.z;
  const int cl = static_cast<int>(blockIdx.x) >> 1;
  g.dh = cl & 1;
  if (MODE == kDQ) {
    const int npairs = (p.q_tiles + 1) >> 1;
    const int sp = npairs - 1 - (cl >> 1);  // heavy causal pairs first
    g.h = blockIdx.y;
    g.kvh = g.h / p.group;
    g.s_head = g.h;
    g.s_row0 = (2 * sp + rank) * kTileRows;
    g.s_limit = p.Nq;
    const int kv_end = p.causal ? min(p.Nkv, (2 * sp + 2) * kTileRows) : p.Nkv;
    g.ncols = (kv_end + kTileRows - 1) / kTileRows;
    g.qt_begin = 0;
    g.nq_h = 0;
    g.rot = g.ncols > 0 ? (2 * sp) % g.ncols : 0;
  } else {
    const int sp = cl >> 1;
    g.kvh = blockIdx.y;
    g.h = g.kvh * p.group;
    g.s_head = g.kvh;
    g.s_row0 = (2 * sp + rank) * kTileRows;
    g.s_limit = p.Nkv;
    g.qt_begin = p.causal ? 2 * sp : 0;  // top-left causal: query rows i >= key row j
    g.nq_h = max(0, p.q_tiles - g.qt_begin);
    g.ncols = p.group * g.nq_h;
    g.rot = g.ncols > 0 ? (2 * sp) % g.ncols : 0;
  }
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

template <int MODE, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                    const __grid_constant__ CUtensorMap map_vh, const __grid_constant__ CUtensorMap map_doh,
                    const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  constexpr bool RES = (MODE == kDV);  // A1 resident
  constexpr int kResBytes = res_bytes(MODE);
  constexpr int kSlotBytes = slot_bytes(MODE);
  const Bars bl = bar_layout(stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kResBytes + stages * kSlotBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  float* stat_sm = reinterpret_cast<float*>(smem + kResBytes + stages * kSlotBytes + 1024);  // dK: [4 warps][2][128]
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t a_sm = smem_u32(smem), ring_sm = a_sm + kResBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const Geo g = make_geo<MODE>(p, static_cast<int>(rank));
  const bool two = (MODE != kDV);  // a second score-like product (dP)
  uint32_t* status = p.status;
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  // stationary A1, A2 (A1 resident for dV); column operands: half-row B1, B2; gradient B3
  const CUtensorMap* mA1 = (MODE == kDQ) ? &map_q : &map_k;
  const CUtensorMap* mA2 = (MODE == kDQ) ? &map_do : &map_v;
  const CUtensorMap* mB1 = (MODE == kDQ) ? &map_kh : &map_qh;
  const CUtensorMap* mB2 = (MODE == kDQ) ? &map_vh : &map_doh;
  const CUtensorMap* mB3 = (MODE == kDV) ? &map_do : ((MODE == kDK) ? &map_q : &map_k);

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar(bl.full + i), 1);
      mbar_init(bar(bl.empty + i), 1);
    }
    mbar_init(bar(bl.a_full), 1);
    mbar_init(bar(bl.x1_full), 1);
    mbar_init(bar(bl.x2_full), 1);
    mbar_init(bar(bl.x1_free), 8);  // four elementwise warps in each CTA
    mbar_init(bar(bl.p_ready), 8);
    mbar_init(bar(bl.acc_ready), 1);
    mbar_init(bar(bl.drain), 1);
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
    // Producer pi issues every nprod-th slot load of this CTA and waits only for
    // its own slot; nprod <= stages keeps parity waits unambiguous.  The bytes
    // of both CTAs' loads are counted on the first CTA's full[s], armed there.
    const int nprod = min(kProducers, stages);
    const int pi = (warp == 0) ? 0 : warp - 1;
    if (lane == 0 && pi < nprod) {
      tma_prefetch_desc(mA1);
      tma_prefetch_desc(mA2);
      tma_prefetch_desc(mB1);
      tma_prefetch_desc(mB2);
      tma_prefetch_desc(mB3);
      if (RES && pi == 0) {
        if (rank == 0) mbar_expect_tx(bar(bl.a_full), 2 * kResBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d_pair(a_sm + c * kChunkBytes, mA1, lead(bl.a_full), c * kChunk, g.s_row0, g.s_head, g.b);
      }
      bool ok = true;
      uint32_t it = 0;
      // kind 0: column half-chunks 4m..4m+3 of B (m = 0, 1); kind 1: stationary
      // chunks 2m, 2m+1 of A with column half-chunks 2m, 2m+1 of B (m = 0..3);
      // kind 2: this CTA's two gradient-operand chunks
      auto slot = [&](int kind, const CUtensorMap* ma, const CUtensorMap* mb, int m, int c) {
        if (ok && static_cast<int>(it % nprod) == pi) {
          const uint32_t s = it % stages, r = it / stages;
          ok = mbar_wait(bar(bl.empty + s), (r & 1) ^ 1, status);
          if (ok) {
            int ch, cr0;
            column<MODE>(g, p, c, &ch, &cr0);
            const uint32_t dst = ring_sm + s * kSlotBytes, fb = lead(bl.full + s);
            const int half_row = cr0 + 64 * static_cast<int>(rank);
            if (kind == 0) {
              if (rank == 0) mbar_expect_tx(bar(bl.full + s), 2 * 4 * kHalfChunkBytes);
              for (int i = 0; i < 4; ++i)
                tma_load_4d_pair(dst + i * kHalfChunkBytes, mb, fb, (4 * m + i) * kChunk, half_row, ch, g.b);
            } else if (kind == 1) {
              if (rank == 0) mbar_expect_tx(bar(bl.full + s), 2 * 2 * (kChunkBytes + kHalfChunkBytes));
              for (int i = 0; i < 2; ++i) {
                tma_load_4d_pair(dst + i * kChunkBytes, ma, fb, (2 * m + i) * kChunk, g.s_row0, g.s_head, g.b);
                tma_load_4d_pair(dst + 2 * kChunkBytes + i * kHalfChunkBytes, mb, fb, (2 * m + i) * kChunk, half_row,
                                 ch, g.b);
              }
            } else {
              if (rank == 0) mbar_expect_tx(bar(bl.full + s), 2 * 2 * kChunkBytes);
              for (int i = 0; i < 2; ++i)
                tma_load_4d_pair(dst + i * kChunkBytes, mB3, fb, (4 * g.dh + 2 * static_cast<int>(rank) + i) * kChunk,
                                 cr0, ch, g.b);
            }
          }
        }
        ++it;
      };
      // Loads follow the MMA thread's order of use: X1 and X2 of column 0, then
      // for each column c: X1 of c + 1, the gradient of c, X2 of c + 1.
      auto x1_loads = [&](int c) {
        if (RES) {
          slot(0, nullptr, mB1, 0, c);
          slot(0, nullptr, mB1, 1, c);
        } else {
          for (int m = 0; m < kChunks / 2; ++m) slot(1, mA1, mB1, m, c);
        }
      };
      auto x2_loads = [&](int c) {
        for (int m = 0; m < kChunks / 2; ++m) slot(1, mA2, mB2, m, c);
      };
      if (g.ncols > 0) {
        x1_loads(0);
        if (two) x2_loads(0);
      }
      for (int c = 0; c < g.ncols && ok; ++c) {
        if (c + 1 < g.ncols) x1_loads(c + 1);
        slot(2, nullptr, nullptr, 0, c);
        if (two && c + 1 < g.ncols) x2_loads(c + 1);
      }
      for (uint32_t s = 0; s < static_cast<uint32_t>(stages) && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / stages) * stages;
        if (static_cast<int>(last % nprod) == pi) mbar_wait(bar(bl.empty + s), (last / stages) & 1, status);
      }
      if (RES && pi == 0 && rank == 0) mbar_wait(bar(bl.a_full), 0, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (first CTA of the pair)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc_x = idesc_f16(BF16, 256, 128, false, false);    // 2 x 128 stationary rows x 128 columns
      const uint32_t idesc_acc = idesc_f16(BF16, 256, 256, false, true);   // 2 x 128 rows x 256 gradient columns
      const uint64_t da = sdesc_sw128(a_sm, 16, 1024);                     // resident A1, K-major
      const uint64_t dk = sdesc_sw128(ring_sm, 16, 1024);                  // ring tiles, K-major
      const uint64_t dm = sdesc_sw128(ring_sm, kChunkBytes, 1024);         // ring tiles, MN-major
      bool ok = RES ? mbar_wait(bar(bl.a_full), 0, status) : true;
      tc_fence_after();
      uint32_t it = 0;
      auto wait_slot = [&]() -> uint32_t {
        const uint32_t s = it % stages;
        ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
        ++it;
        tc_fence_after();
        return s;
      };
      // X (+)= A B^T over the eight chunks, A and B streamed: chunks 2m, 2m+1 of
      // both in slot m
      auto product_streamed = [&](uint32_t x_tm) {
        for (int m = 0; m < kChunks / 2 && ok; ++m) {
          const uint32_t s = wait_slot();
          if (!ok) return;
          for (int i = 0; i < 2; ++i) {
            const int c = 2 * m + i;
            const uint64_t a = sdesc_advance(dk, s * kSlotBytes + i * kChunkBytes);
            const uint64_t bd = sdesc_advance(dk, s * kSlotBytes + 2 * kChunkBytes + i * kHalfChunkBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_pair(x_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x, (c | kk) != 0);
          }
          umma_commit_pair(bar(bl.empty + s), 3);
        }
      };
      // X1 (+)= A1 B1^T over the eight chunks: with A1 resident (dV), B1
      // half-chunks in two slots; otherwise both streamed
      auto product1 = [&]() {
        if constexpr (!RES) {
          product_streamed(tbase + kX1);
        } else {
          for (int m = 0; m < 2 && ok; ++m) {
            const uint32_t s = wait_slot();
            if (!ok) return;
            for (int i = 0; i < 4; ++i) {
              const int c = 4 * m + i;
              const uint64_t a = sdesc_advance(da, c * kChunkBytes);
              const uint64_t bd = sdesc_advance(dk, s * kSlotBytes + i * kHalfChunkBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss_pair(tbase + kX1, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x,
                             (c | kk) != 0);
            }
            umma_commit_pair(bar(bl.empty + s), 3);
          }
        }
      };
      auto product2 = [&]() { product_streamed(tbase + kX2); };
      // X1 is read only by the elementwise warps, which free it before computing
      // P and dS; X2 ends up holding P or dS, the A operand of the gradient.  So
      // the next column's X1 product overlaps this column's elementwise work,
      // and X2 is rewritten by the next product right after the gradient MMAs.
      // X1 and X2 each signal their own barrier, so the elementwise warps copy
      // the scores out (and free X1) while the gradient and dP MMAs still run.
      if (g.ncols > 0) {
        product1();
        if (ok) umma_commit_pair(bar(bl.x1_full), 3);
        if (two && ok) product2();
        if (two && ok) umma_commit_pair(bar(bl.x2_full), 3);
      }
      for (int c = 0; c < g.ncols && ok; ++c) {
        const bool more = c + 1 < g.ncols;
        if (more) {
          ok = mbar_wait(bar(bl.x1_free), c & 1, status);
          if (!ok) break;
          tc_fence_after();
          product1();
          if (!ok) break;
          umma_commit_pair(bar(bl.x1_full), 3);
        }
        ok = mbar_wait(bar(bl.p_ready), c & 1, status);
        if (!ok) break;
        tc_fence_after();
        {
          const uint32_t s = wait_slot();
          if (!ok) break;
          const uint64_t bd = sdesc_advance(dm, s * kSlotBytes);
          const uint32_t acc0 = c > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts_pair(tbase, tbase + kX2 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_acc, acc0 | (kk > 0));
          umma_commit_pair(bar(bl.empty + s), 3);
        }
        umma_commit_pair(bar(bl.acc_ready), 3);
        if (more && two) {
          // X2 still holds dS of this column, read by the gradient MMAs just
          // issued; MMAs issued by one thread execute in issue order, so the
          // next column's X2 product may follow them without a wait.
          product2();
          if (!ok) break;
          umma_commit_pair(bar(bl.x2_full), 3);
        }
      }
      umma_commit_pair(bar(bl.drain), 1);
      mbar_wait(bar(bl.drain), 0, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise + epilogue
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int r = tid - 128;
    const int srow = g.s_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t x1_free_lead = lead(bl.x1_free), p_ready_lead = lead(bl.p_ready);
    float lse2_row = 0.f, delta_row = 0.f;
    if (MODE == kDQ) {
      const int64_t idx = (static_cast<int64_t>(g.b) * p.Hq + g.h) * p.Nq + min(srow, p.Nq - 1);
      lse2_row = p.lse2[idx];
      delta_row = p.delta[idx];
    }
    bool ok = true;
    auto arrive_lead = [&](uint32_t a) {
      if (rank == 0)
        mbar_arrive(a);
      else
        mbar_arrive_remote(a);
    };
    auto chunk = [&](uint32_t col, int c4, float (&f)[32]) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_off + col + c4 * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    };
    for (int c = 0; c < g.ncols; ++c) {
      int ch, cr0;
      column<MODE>(g, p, c, &ch, &cr0);
      // Column statistics (dV, dK): lane l of every warp loads lse2 and Delta of
      // column rows cr0 + l + 32 c4.  dV's threads take theirs with shuffles;
      // dK's warps stage them in their own 1 KB of shared memory and read them
      // back four at a time with broadcast loads (a quarter of the shuffle
      // traffic, which shares the shared-memory pipe with the MMA operands).
      float l2v[4] = {0.f, 0.f, 0.f, 0.f}, dlv[4] = {0.f, 0.f, 0.f, 0.f};
      float* wst = stat_sm + (warp - 4) * 256;  // dK: [lse2 x 128 | Delta x 128] of this warp
      if (MODE != kDQ) {
        const int64_t sbase = (static_cast<int64_t>(g.b) * p.Hq + ch) * p.Nq;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int64_t i = sbase + min(cr0 + c4 * 32 + lane, p.Nq - 1);
          l2v[c4] = p.lse2[i];
          if (two) dlv[c4] = p.delta[i];
        }
        if constexpr (MODE == kDK) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            wst[c4 * 32 + lane] = l2v[c4];
            wst[128 + c4 * 32 + lane] = dlv[c4];
          }
          __syncwarp();
        }
      }
      const float4* wst4 = reinterpret_cast<const float4*>(wst);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x1_full), c & 1, status));
      if (!ok) break;
      tc_fence_after();
      float pv[128];
      bool plain;
      if (MODE == kDQ)
        plain = srow < p.Nq && cr0 + kTileRows <= p.Nkv && (!p.causal || cr0 + kTileRows - 1 <= srow) &&
                lse2_row > -INFINITY;
      else
        plain = srow < p.Nkv && cr0 + kTileRows <= p.Nq && (!p.causal || srow <= cr0);
      plain = __all_sync(0xffffffffu, plain) && p.bias == nullptr;
      // Copy the raw scores out of TMEM first and free X1 at once, so the next
      // column's score product runs while this thread computes the exponentials
      // (they are limited by the special-function unit's throughput).
      uint32_t raw0[32], raw1[32], raw2[32], raw3[32];
      tmem_ld32(tbase + lane_off + kX1, raw0);
      tmem_ld32(tbase + lane_off + kX1 + 32, raw1);
      tmem_ld32(tbase + lane_off + kX1 + 64, raw2);
      tmem_ld32(tbase + lane_off + kX1 + 96, raw3);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        pv[e] = __uint_as_float(raw0[e]);
        pv[32 + e] = __uint_as_float(raw1[e]);
        pv[64 + e] = __uint_as_float(raw2[e]);
        pv[96 + e] = __uint_as_float(raw3[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(x1_free_lead);
      if (MODE == kDK && plain) {
#pragma unroll
        for (int e4 = 0; e4 < 32; ++e4) {
          const float4 l2 = wst4[e4];
          pv[4 * e4 + 0] = ex2(fmaf(pv[4 * e4 + 0], p.scale_log2, -l2.x));
          pv[4 * e4 + 1] = ex2(fmaf(pv[4 * e4 + 1], p.scale_log2, -l2.y));
          pv[4 * e4 + 2] = ex2(fmaf(pv[4 * e4 + 2], p.scale_log2, -l2.z));
          pv[4 * e4 + 3] = ex2(fmaf(pv[4 * e4 + 3], p.scale_log2, -l2.w));
        }
      } else if (plain) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float l2 = (MODE == kDQ) ? lse2_row : __shfl_sync(0xffffffffu, l2v[c4], e);
            pv[c4 * 32 + e] = ex2(fmaf(pv[c4 * 32 + e], p.scale_log2, -l2));
          }
        }
      } else {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int ci = c4 * 32 + e;
            int i, j, ic;
            float l2;
            if (MODE == kDQ) {
              i = srow;
              j = cr0 + ci;
              ic = min(i, p.Nq - 1);
              l2 = lse2_row;
            } else {
              i = cr0 + ci;
              j = srow;
              ic = min(i, p.Nq - 1);
              l2 = (MODE == kDK) ? wst[ci] : __shfl_sync(0xffffffffu, l2v[c4], e);
            }
            const int hq = (MODE == kDQ) ? g.h : ch;
            const bool valid = i < p.Nq && j < p.Nkv && !(p.causal && j > i) && l2 > -INFINITY;
            float xv = fmaf(pv[ci], p.scale_log2, -l2);
            if (p.bias)
              xv = fmaf(__ldg(p.bias + g.b * p.bias_sb + hq * p.bias_sh + static_cast<int64_t>(ic) * p.bias_sq +
                              static_cast<int64_t>(min(j, p.Nkv - 1)) * p.bias_sk),
                        kLog2e, xv);
            pv[ci] = valid ? ex2(xv) : 0.f;
          }
        }
      }
      if (two) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x2_full), c & 1, status));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float f[32];
          chunk(kX2, c4, f);
          if constexpr (MODE == kDK) {
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 dl = wst4[32 + c4 * 8 + e4];
              pv[c4 * 32 + 4 * e4 + 0] *= f[4 * e4 + 0] - dl.x;
              pv[c4 * 32 + 4 * e4 + 1] *= f[4 * e4 + 1] - dl.y;
              pv[c4 * 32 + 4 * e4 + 2] *= f[4 * e4 + 2] - dl.z;
              pv[c4 * 32 + 4 * e4 + 3] *= f[4 * e4 + 3] - dl.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int ci = c4 * 32 + e;
              const float dl = (MODE == kDQ) ? delta_row : __shfl_sync(0xffffffffu, dlv[c4], e);
              pv[ci] = pv[ci] * (f[e] - dl);
            }
          }
        }
      }
      {
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          lo[e] = pack2<BF16>(pv[2 * e], pv[2 * e + 1]);
          hi[e] = pack2<BF16>(pv[64 + 2 * e], pv[64 + 2 * e + 1]);
        }
        if (!two && c > 0) {
          // X2 held the previous column's P, read by its gradient MMAs (with
          // dP, the X2 product of this column already waited for them).
          ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready), (c - 1) & 1, status));
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st32(tbase + lane_off + kX2, lo);
        tmem_st32(tbase + lane_off + kX2 + 32, hi);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_lead(p_ready_lead);
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      if (g.ncols > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready), (g.ncols - 1) & 1, status));
        if (ok) tc_fence_after();
      }
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
        for (int oc = 0; oc < 4; ++oc) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            if (g.ncols > 0) {
              tmem_ld32(tbase + lane_off + oc * kChunk + hh * 32, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (srow < g.s_limit) {
              uint4* dst = reinterpret_cast<uint4*>(orow + (4 * g.dh + oc) * kChunk + hh * 32);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 w;
                w.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]) * mul, __uint_as_float(v[8 * q4 + 1]) * mul);
                w.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]) * mul, __uint_as_float(v[8 * q4 + 3]) * mul);
                w.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]) * mul, __uint_as_float(v[8 * q4 + 5]) * mul);
                w.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]) * mul, __uint_as_float(v[8 * q4 + 7]) * mul);
                dst[q4] = w;
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

template <int MODE, bool BF16>
cudaError_t launch_mode(const BwdParams& p_in, const BwdMaps& m, cudaStream_t st) {
  BwdParams p = p_in;
  constexpr int kMaxSmem = 232448;
  int stages = (kMaxSmem - smem_bytes(MODE, 0)) / slot_bytes(MODE);
  stages = min(stages, 4);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  p.slot_chunks = slot_bytes(MODE) / kChunkBytes;
  const int smem = smem_bytes(MODE, stages);
  auto kern = bwd_pair_kernel<MODE, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (MODE == kDQ) ? p.q_tiles : p.kv_tiles;
  const int npairs = (tiles + 1) / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = (MODE == kDQ) ? dim3(4 * npairs, p.Hq, p.B) : dim3(4 * npairs, p.Hkv, p.B);
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
cudaError_t launch_modes(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  cudaError_t e;
  if ((e = launch_mode<kDV, BF16>(p, m, st)) != cudaSuccess) return e;
  if ((e = launch_mode<kDK, BF16>(p, m, st)) != cudaSuccess) return e;
  return launch_mode<kDQ, BF16>(p, m, st);
}

}  // namespace

bool bwd_pair_supported(const BwdParams& p) { return p.n_chunks == kChunks; }

cudaError_t launch_bwd_pair(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_modes<true>(p, m, s) : launch_modes<false>(p, m, s);
}

}  // namespace ffpa
