// Attention backward for large head dimensions on sm_103a.
//
// The FFPA Attention Benchmark page ("More Benchmark") describes the SM100
// backward as four launches, preprocess, dV, dK and dQ, executing 8 GEMM
// passes.  This file builds the same decomposition:
//   preprocess:  Delta_i = sum_d dO_id O_id,  lse2_i = lse_i * log2(e)
//   dV  (per key tile):   S^T = K Q^T;  P^T = 2^(S^T c + bias2 - lse2);  dV += P^T dO        (2 GEMMs)
//   dK  (per key tile):   S^T, dP^T = V dO^T;  dS^T = P^T (dP^T - Delta);  dK += dS^T Q    (3 GEMMs)
//   dQ  (per query tile): S = Q K^T, dP = dO V^T;  dS = P (dP - Delta);  dQ += dS K        (3 GEMMs)
// with c = scale * log2(e), and dK, dQ scaled by `scale` in the epilogue.
// P is rebuilt exactly from the forward's lse, so no online softmax is needed.
//
// Each kernel keeps one 128-row tile "stationary" (key rows for dV/dK, query
// rows for dQ) and sweeps the other side in 128-row "column" tiles; one CTA
// computes the score tiles over all of D with tcgen05.mma into TMEM and
// accumulates the whole gradient (<= 256 TMEM columns).  GQA: the dV/dK
// kernels sweep every query head of the group, so the group's sum forms in
// TMEM without any atomics or workspace.
//
// These kernels serve D <= 256.  launch_bwd hands larger head dimensions,
// after the preprocess, to the fused dK/dV cluster kernel of bwd_xch.cu and
// then to the dQ kernel of bwd_dq.cu (D = 320 .. 512) or bwd_xch.cu's dQ mode
// (D = 576 .. 1024).
//
// TMEM (512 columns): gradient accumulator [0, 256), X1 [256, 384) (scores),
// X2 [384, 512) (dP, then P or dS as the bf16/f16 A operand of the gradient).
// Warp roles: warps 0, 2, 3 TMA producers, warp 1 TMEM owner + MMA issuer,
// warps 4-7 elementwise + epilogue (thread = stationary row = TMEM lane).
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
constexpr int kMaxAccChunks = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct Bars {
  int full, empty, a_full, x_full, x1_free, p_ready, acc_ready, acc_free, drain, count;
};
__host__ __device__ inline Bars bar_layout(int stages) {
  Bars b;
  b.full = 0;
  b.empty = stages;
  b.a_full = 2 * stages;
  b.x_full = b.a_full + 1;
  b.x1_free = b.x_full + 1;
  b.p_ready = b.x1_free + 1;
  b.acc_ready = b.p_ready + 1;
  b.acc_free = b.acc_ready + 1;
  b.drain = b.acc_free + 1;
  b.count = b.drain + 1;
  return b;
}

struct Plan {
  int a_chunks;  // chunks the score products reduce over (per resident operand)
  int n_a;       // resident stationary operands (A1, then A2); the rest stream through the ring
  int a_off, ring_off, bar_off, total;
};
__host__ __device__ inline Plan make_plan(int n_chunks, int stages, int n_res, int slot_chunks) {
  Plan s;
  s.a_chunks = n_chunks;
  s.n_a = n_res;
  s.a_off = 0;
  s.ring_off = s.n_a * s.a_chunks * kChunkBytes;
  s.bar_off = s.ring_off + stages * slot_chunks * kChunkBytes;
  s.total = s.bar_off + 1024;
  return s;
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

// Preprocess: one warp per query row.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __grid_constant__ BwdParams p) {
  typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Nq;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int i = static_cast<int>(row % p.Nq);
  const int h = static_cast<int>((row / p.Nq) % p.Hq);
  const int b = static_cast<int>(row / (static_cast<int64_t>(p.Nq) * p.Hq));
  const T* o = reinterpret_cast<const T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(i) * p.o_sn;
  const T* d = reinterpret_cast<const T*>(p.dout) + b * p.do_sb + h * p.do_sh + static_cast<int64_t>(i) * p.do_sn;
  float acc = 0.f;
  for (int c = lane * 8; c < p.D; c += 256) {
    const uint4 uo = __ldg(reinterpret_cast<const uint4*>(o + c));
    const uint4 ud = __ldg(reinterpret_cast<const uint4*>(d + c));
    const uint32_t wo[4] = {uo.x, uo.y, uo.z, uo.w}, wd[4] = {ud.x, ud.y, ud.z, ud.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 fo, fd;
      if constexpr (BF16) {
        fo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wo[e]));
        fd = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[e]));
      } else {
        fo = __half22float2(*reinterpret_cast<const __half2*>(&wo[e]));
        fd = __half22float2(*reinterpret_cast<const __half2*>(&wd[e]));
      }
      acc = fmaf(fo.x, fd.x, acc);
      acc = fmaf(fo.y, fd.y, acc);
    }
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    p.delta[row] = acc;
    p.lse2[row] = p.lse[row] * kLog2e;
  }
}

// Stationary/column geometry of one CTA.
struct Geo {
  int b, h, kvh;      // batch, query head (dQ) and kv head
  int s_head, s_row0; // stationary tile: head index in its tensor, first row
  int s_limit;        // rows of the stationary tensor (Nkv for dV/dK, Nq for dQ)
  int qt_begin, nq_h; // dV/dK: first query tile and query tiles per head
  int ncols;          // column tiles
  int rot;            // column sweep starts here (stationary tiles start at different columns)
};

template <int MODE>
__device__ __forceinline__ Geo make_geo(const BwdParams& p) {
  Geo g;
  g.b = blockIdx.z;
  if (MODE == kDQ) {
    const int qt = p.q_tiles - 1 - static_cast<int>(blockIdx.x);  // heavy causal tiles first
    g.h = blockIdx.y;
    g.kvh = g.h / p.group;
    g.s_head = g.h;
    g.s_row0 = qt * kTileRows;
    g.s_limit = p.Nq;
    const int kv_end = p.causal ? min(p.Nkv, g.s_row0 + kTileRows) : p.Nkv;
    g.ncols = (kv_end + kTileRows - 1) / kTileRows;
    g.qt_begin = 0;
    g.nq_h = 0;
    g.rot = g.ncols > 0 ? qt % g.ncols : 0;
  } else {
    const int kvt = static_cast<int>(blockIdx.x);
    g.kvh = blockIdx.y;
    g.h = g.kvh * p.group;
    g.s_head = g.kvh;
    g.s_row0 = kvt * kTileRows;
    g.s_limit = p.Nkv;
    g.qt_begin = p.causal ? kvt : 0;  // top-left causal: query rows i >= key row j
    g.nq_h = max(0, p.q_tiles - g.qt_begin);
    g.ncols = p.group * g.nq_h;
    g.rot = g.ncols > 0 ? kvt % g.ncols : 0;
  }
  return g;
}

// Column tile c -> (head, first row) in the column tensor.
template <int MODE>
__device__ __forceinline__ void column(const Geo& g, const BwdParams& p, int c, int* head, int* row0) {
  // Concurrent CTAs of a head would otherwise stream the same column tiles at
  // the same time; starting each sweep at a different tile spreads the reads.
  // The gradient is a sum over columns, so the order does not change it.
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
    bwd_main_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ BwdParams p, const int n_res) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  const int G = p.slot_chunks;  // 16 KB tiles per ring slot
  const uint32_t slot_bytes = G * kChunkBytes;
  const Plan plan = make_plan(p.n_chunks, stages, n_res, G);
  const Bars bl = bar_layout(stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t s_base = smem_u32(smem);
  const uint32_t a_sm = s_base + plan.a_off, ring_sm = s_base + plan.ring_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Geo g = make_geo<MODE>(p);
  const int n = p.n_chunks;
  // the score products reduce over chunks s0 .. s0 + s_n - 1 and the gradient
  // covers chunks own0 .. own0 + own_n - 1: all of D
  const int s0 = 0, s_n = n, own0 = 0, own_n = n;
  const int passes = (n + kMaxAccChunks - 1) / kMaxAccChunks;
  const bool two = (MODE != kDV);  // a second score-like product (dP)
  uint32_t* status = p.status;

  const CUtensorMap* mA1 = (MODE == kDQ) ? &map_q : &map_k;
  const CUtensorMap* mA2 = (MODE == kDQ) ? &map_do : &map_v;
  const CUtensorMap* mB1 = (MODE == kDQ) ? &map_k : &map_q;
  const CUtensorMap* mB2 = (MODE == kDQ) ? &map_v : &map_do;
  const CUtensorMap* mB3 = (MODE == kDV) ? &map_do : ((MODE == kDK) ? &map_q : &map_k);

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar(bl.full + i), 1);
      mbar_init(bar(bl.empty + i), 1);
    }
    mbar_init(bar(bl.a_full), 1);
    mbar_init(bar(bl.x_full), 1);
    mbar_init(bar(bl.x1_free), 4);
    mbar_init(bar(bl.p_ready), 4);
    mbar_init(bar(bl.acc_ready), 1);
    mbar_init(bar(bl.acc_free), 4);
    mbar_init(bar(bl.drain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 || warp == 2 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // Three warps (one lane each) issue the ring loads: producer pi owns every
    // nprod-th load and waits only for its own slot to be released. Arming
    // a barrier and issuing a TMA load blocks the issuing thread for ~500
    // cycles, so one thread alone cannot keep the ring full, and lanes of one
    // warp would have to wait for one another's slots.
    // A parity wait tells apart only the current and the previous phase of a
    // barrier, so no producer may run two rounds ahead of a slot's barrier:
    // producer pi waits for load i - stages before issuing load i, having
    // issued load i - nprod, which needs nprod <= stages.
    const int nprod = min(kProducers, stages);
    const int pi = (warp == 0) ? 0 : warp - 1;
    if (lane == 0 && pi < nprod) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      tma_prefetch_desc(&map_do);
      if (pi == 0 && n_res > 0) {
        mbar_expect_tx(bar(bl.a_full), n_res * s_n * kChunkBytes);
        for (int c = 0; c < s_n; ++c) {
          tma_load_4d(a_sm + c * kChunkBytes, mA1, bar(bl.a_full), (s0 + c) * kChunk, g.s_row0, g.s_head, g.b);
          if (n_res > 1)
            tma_load_4d(a_sm + (plan.a_chunks + c) * kChunkBytes, mA2, bar(bl.a_full), (s0 + c) * kChunk,
                        g.s_row0, g.s_head, g.b);
        }
      }
      bool ok = true;
      uint32_t it = 0;
      // One ring slot holds up to G 16 KB tiles loaded under a single barrier
      // phase: each phase of a slot (arm, land, wait, release) costs the SM a
      // few hundred cycles whatever its size, so two tiles per phase move
      // nearly twice the bytes of one.  Tile i of the slot is (m[i], chunk
      // dc[i], rows from row[i], head hd[i]).
      auto load = [&](int cn, const CUtensorMap* const* m, const int* dc, const int* row, const int* hd) {
        if (ok && static_cast<int>(it % nprod) == pi) {
          const uint32_t s = it % stages, r = it / stages;
          ok = mbar_wait(bar(bl.empty + s), (r & 1) ^ 1, status);
          if (ok) {
            mbar_expect_tx(bar(bl.full + s), cn * kChunkBytes);
            for (int i = 0; i < cn; ++i)
              tma_load_4d(ring_sm + s * slot_bytes + i * kChunkBytes, m[i], bar(bl.full + s), dc[i] * kChunk, row[i],
                          hd[i], g.b);
          }
        }
        ++it;
      };
      // cn consecutive chunks of one operand
      auto load_run = [&](const CUtensorMap* m, int c0, int cn, int row, int head) {
        const CUtensorMap* ms[2] = {m, m};
        const int dc[2] = {c0, c0 + 1}, rw[2] = {row, row}, hd[2] = {head, head};
        load(cn, ms, dc, rw, hd);
      };
      // A score product over the chunks s0 .. s0+s_n-1: with A resident only B
      // streams (G chunks per slot); otherwise chunk cc of A and of B share a
      // slot (G = 2) or take one slot each (G = 1).
      auto product_loads = [&](const CUtensorMap* mA, bool a_res, const CUtensorMap* mB, int c) {
        int ch, cr0;
        column<MODE>(g, p, c, &ch, &cr0);
        if (a_res) {
          for (int cc = 0; cc < s_n; cc += G) load_run(mB, s0 + cc, min(G, s_n - cc), cr0, ch);
        } else if (G == 2) {
          for (int cc = 0; cc < s_n; ++cc) {
            const CUtensorMap* ms[2] = {mA, mB};
            const int dc[2] = {s0 + cc, s0 + cc}, rw[2] = {g.s_row0, cr0}, hd[2] = {g.s_head, ch};
            load(2, ms, dc, rw, hd);
          }
        } else {
          for (int cc = 0; cc < s_n; ++cc) {
            load_run(mA, s0 + cc, 1, g.s_row0, g.s_head);
            load_run(mB, s0 + cc, 1, cr0, ch);
          }
        }
      };
      // Loads follow the MMA warp's order of use: X1 and X2 of column 0, then
      // for each column c: X1 of c + 1, the gradient of c, X2 of c + 1.
      auto x1_loads = [&](int c) { product_loads(mA1, n_res >= 1, mB1, c); };
      auto x2_loads = [&](int c) { product_loads(mA2, n_res >= 2, mB2, c); };
      for (int pass = 0; pass < passes && ok; ++pass) {
        const int oc0 = pass * kMaxAccChunks;
        const int oc_n = max(0, min(kMaxAccChunks, own_n - oc0));
        if (g.ncols > 0) {
          x1_loads(0);
          if (two) x2_loads(0);
        }
        for (int c = 0; c < g.ncols && ok; ++c) {
          if (c + 1 < g.ncols) x1_loads(c + 1);
          int ch, cr0;
          column<MODE>(g, p, c, &ch, &cr0);
          for (int oc = 0; oc < oc_n; oc += G) load_run(mB3, own0 + oc0 + oc, min(G, oc_n - oc), cr0, ch);
          if (two && c + 1 < g.ncols) x2_loads(c + 1);
        }
      }
      // Wait for the last release of each ring slot whose last load was ours:
      // the MMA warp's commit arrives on empty[s] only when the MMAs reading the
      // slot are done, and commit arrivals are not ordered with respect to one
      // another, so one still in flight at exit would land in the next CTA's
      // shared memory. (After a timeout `it` stops short; the waits stay bounded.)
      for (uint32_t s = 0; s < static_cast<uint32_t>(stages) && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / stages) * stages;
        if (static_cast<int>(last % nprod) == pi) mbar_wait(bar(bl.empty + s), (last / stages) & 1, status);
      }
      if (pi == 0 && n_res > 0) mbar_wait(bar(bl.a_full), 0, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are formed once and advanced by constants (building them per
    // MMA made the issuing thread the bottleneck).
    if (lane == 0) {
      const uint32_t idesc_x = idesc_f16(BF16, 128, 128, false, false);
      const uint32_t idesc_acc = idesc_f16(BF16, 128, 64, false, true);
      const uint32_t idesc_acc2 = idesc_f16(BF16, 128, 128, false, true);  // two chunks in adjacent slots
      const uint64_t da = sdesc_sw128(a_sm, 16, 1024);                     // resident operands, K-major
      const uint64_t dk = sdesc_sw128(ring_sm, 16, 1024);                  // ring slots, K-major
      const uint64_t dm = sdesc_sw128(ring_sm, kChunkBytes, 1024);         // ring slots, MN-major
      bool ok = n_res > 0 ? mbar_wait(bar(bl.a_full), 0, status) : true;
      tc_fence_after();
      uint32_t it = 0;
      int t0 = 0;
      // one score-like product: X (+)= A B^T over the chunks s0 .. s0+s_n-1,
      // consuming the ring in the producer's order (see product_loads)
      auto product = [&](uint32_t x_tm, int a_slot) {
        const bool resident = a_slot < n_res;
        if (resident) {
          for (int cc = 0; cc < s_n && ok; cc += G) {
            const uint32_t sb = it % stages;
            ok = mbar_wait(bar(bl.full + sb), (it / stages) & 1, status);
            if (!ok) return;
            ++it;
            tc_fence_after();
            const int cn = min(G, s_n - cc);
            for (int i = 0; i < cn; ++i) {
              const uint64_t a = sdesc_advance(da, (a_slot * plan.a_chunks + cc + i) * kChunkBytes);
              const uint64_t bd = sdesc_advance(dk, sb * slot_bytes + i * kChunkBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss(x_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x, ((cc + i) | kk) != 0);
            }
            umma_commit(bar(bl.empty + sb));
          }
          return;
        }
        for (int cc = 0; cc < s_n && ok; ++cc) {
          uint64_t a, bd;
          uint32_t sa = 0, sb;
          if (G == 2) {  // A and B chunk in one slot
            sb = it % stages;
            ok = mbar_wait(bar(bl.full + sb), (it / stages) & 1, status);
            if (!ok) return;
            ++it;
            a = sdesc_advance(dk, sb * slot_bytes);
            bd = sdesc_advance(dk, sb * slot_bytes + kChunkBytes);
          } else {
            sa = it % stages;
            ok = mbar_wait(bar(bl.full + sa), (it / stages) & 1, status);
            if (!ok) return;
            ++it;
            sb = it % stages;
            ok = mbar_wait(bar(bl.full + sb), (it / stages) & 1, status);
            if (!ok) return;
            ++it;
            a = sdesc_advance(dk, sa * kChunkBytes);
            bd = sdesc_advance(dk, sb * kChunkBytes);
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_ss(x_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_x, (cc | kk) != 0);
          if (G == 1) umma_commit(bar(bl.empty + sa));
          umma_commit(bar(bl.empty + sb));
        }
      };
      for (int pass = 0; pass < passes && ok; ++pass) {
        const int oc_n = max(0, min(kMaxAccChunks, own_n - pass * kMaxAccChunks));
        // With no columns the MMAs never touch the accumulator, and the epilogue
        // may already have arrived for several passes (a parity wait would then
        // alias), so there is nothing to wait for.
        if (pass > 0 && g.ncols > 0) {
          ok = mbar_wait(bar(bl.acc_free), (pass - 1) & 1, status);
          tc_fence_after();
        }
        // X1 (scores) is read only by the elementwise warps, which free it before
        // computing P and dS; X2 ends up holding P or dS, the A operand of the
        // gradient MMAs.  So the next column's X1 product overlaps this
        // column's elementwise work, and X2 is rewritten only after the
        // gradient MMAs reading it have completed (tcgen05.mma does not order a
        // later write of D after an earlier read of A in TMEM).
        if (g.ncols > 0) {
          product(tbase + kX1, 0);
          if (two && ok) product(tbase + kX2, 1);
          if (ok) umma_commit(bar(bl.x_full));
        }
        for (int c = 0; c < g.ncols && ok; ++c) {
          const int t = t0 + c;
          const bool more = c + 1 < g.ncols;
          if (more) {
            ok = mbar_wait(bar(bl.x1_free), t & 1, status);
            if (!ok) break;
            tc_fence_after();
            product(tbase + kX1, 0);
            if (!ok) break;
            if (!two) umma_commit(bar(bl.x_full));
          }
          ok = mbar_wait(bar(bl.p_ready), t & 1, status);
          if (!ok) break;
          tc_fence_after();
          // gradient += (P or dS) B3: two chunks per MMA (N=128) when they share a
          // ring slot, or (one chunk per slot) sit in adjacent slots
          for (int oc = 0; oc < oc_n && ok;) {
            const uint32_t s = it % stages;
            if (G == 2) {
              ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
              if (!ok) break;
              tc_fence_after();
              const uint64_t bd = sdesc_advance(dm, s * slot_bytes);
              const uint32_t acc0 = c > 0 ? 1u : 0u;
              const uint32_t idesc = (oc + 1 < oc_n) ? idesc_acc2 : idesc_acc;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + oc * kChunk, tbase + kX2 + kk * 8, sdesc_advance(bd, kk * 2048), idesc,
                        acc0 | (kk > 0));
              umma_commit(bar(bl.empty + s));
              it += 1;
              oc += 2;
              continue;
            }
            const bool pair = (oc + 1 < oc_n) && (s + 1 < static_cast<uint32_t>(stages));
            ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
            if (ok && pair) ok = mbar_wait(bar(bl.full + s + 1), ((it + 1) / stages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bd = sdesc_advance(dm, s * kChunkBytes);
            const uint32_t acc0 = c > 0 ? 1u : 0u;
            if (pair) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + oc * kChunk, tbase + kX2 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_acc2,
                        acc0 | (kk > 0));
              umma_commit(bar(bl.empty + s));
              umma_commit(bar(bl.empty + s + 1));
              it += 2;
              oc += 2;
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + oc * kChunk, tbase + kX2 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_acc,
                        acc0 | (kk > 0));
              umma_commit(bar(bl.empty + s));
              it += 1;
              oc += 1;
            }
          }
          if (!ok) break;
          umma_commit(bar(bl.acc_ready));
          if (more && two) {
            ok = mbar_wait(bar(bl.acc_ready), t & 1, status);
            if (!ok) break;
            tc_fence_after();
            product(tbase + kX2, 1);
            if (!ok) break;
            umma_commit(bar(bl.x_full));
          }
        }
        t0 += g.ncols;
      }
      umma_commit(bar(bl.drain));
      mbar_wait(bar(bl.drain), 0, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ elementwise + epilogue
    typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
    const int r = tid - 128;
    const int srow = g.s_row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    float lse2_row = 0.f, delta_row = 0.f;
    if (MODE == kDQ) {
      const int64_t idx = (static_cast<int64_t>(g.b) * p.Hq + g.h) * p.Nq + min(srow, p.Nq - 1);
      lse2_row = p.lse2[idx];
      delta_row = p.delta[idx];
    }
    bool ok = true;
    int t0 = 0;
    // 32 columns of a score tile
    auto chunk = [&](uint32_t col, int c4, float (&f)[32]) {
      uint32_t v[32];
      tmem_ld32(tbase + lane_off + col + c4 * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
    };
    for (int pass = 0; pass < passes && ok; ++pass) {
      const int oc0 = pass * kMaxAccChunks;
      const int oc_n = max(0, min(kMaxAccChunks, own_n - oc0));
      for (int c = 0; c < g.ncols; ++c) {
        const int t = t0 + c;
        int ch, cr0;
        column<MODE>(g, p, c, &ch, &cr0);
        // Column statistics (dV, dK): lane l of every warp loads lse2 and Delta
        // of column rows cr0 + l + 32 c4; each thread then takes the values it
        // needs with warp shuffles instead of one dependent global load per
        // score.  The loads are issued before the wait so their latency hides.
        float l2v[4] = {0.f, 0.f, 0.f, 0.f}, dlv[4] = {0.f, 0.f, 0.f, 0.f};
        if (MODE != kDQ) {
          const int64_t sbase = (static_cast<int64_t>(g.b) * p.Hq + ch) * p.Nq;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int64_t i = sbase + min(cr0 + c4 * 32 + lane, p.Nq - 1);
            l2v[c4] = p.lse2[i];
            if (two) dlv[c4] = p.delta[i];
          }
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.x_full), t & 1, status));
        if (!ok) break;
        tc_fence_after();
        float pv[128];
        // A tile with no masked score and no bias (every tile but the diagonal
        // and the ragged edges) skips the per-score checks.
        bool plain;
        if (MODE == kDQ)
          plain = srow < p.Nq && cr0 + kTileRows <= p.Nkv && (!p.causal || cr0 + kTileRows - 1 <= srow) &&
                  lse2_row > -INFINITY;
        else
          plain = srow < p.Nkv && cr0 + kTileRows <= p.Nq && (!p.causal || srow <= cr0);
        plain = __all_sync(0xffffffffu, plain) && p.bias == nullptr;
        if (plain) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float f[32];
            chunk(kX1, c4, f);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float l2 = (MODE == kDQ) ? lse2_row : __shfl_sync(0xffffffffu, l2v[c4], e);
              pv[c4 * 32 + e] = ex2(fmaf(f[e], p.scale_log2, -l2));
            }
          }
        } else {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float f[32];
          chunk(kX1, c4, f);
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
              l2 = __shfl_sync(0xffffffffu, l2v[c4], e);
            }
            const int hq = (MODE == kDQ) ? g.h : ch;
            const bool valid = i < p.Nq && j < p.Nkv && !(p.causal && j > i) && l2 > -INFINITY;
            float xv = fmaf(f[e], p.scale_log2, -l2);
            if (p.bias)
              xv = fmaf(__ldg(p.bias + g.b * p.bias_sb + hq * p.bias_sh + static_cast<int64_t>(ic) * p.bias_sq +
                              static_cast<int64_t>(min(j, p.Nkv - 1)) * p.bias_sk),
                        kLog2e, xv);
            pv[ci] = valid ? ex2(xv) : 0.f;
          }
        }
        }
        // The scores have been read: X1 may take the next column's.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bl.x1_free));
        if (two) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float f[32];
            chunk(kX2, c4, f);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int ci = c4 * 32 + e;
              float dl;
              if (MODE == kDQ)
                dl = delta_row;
              else
                dl = __shfl_sync(0xffffffffu, dlv[c4], e);
              pv[ci] = pv[ci] * (f[e] - dl);
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
          if (!two && t > 0) {
            // X2 held the previous column's P, read by its gradient MMAs (with
            // dP, the X2 product of this column already waited for them).
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready), (t - 1) & 1, status));
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st32(tbase + lane_off + kX2, lo);
          tmem_st32(tbase + lane_off + kX2 + 32, hi);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bl.p_ready));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (g.ncols > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.acc_ready), (t0 + g.ncols - 1) & 1, status));
        if (!ok) break;
        tc_fence_after();
      }
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
      for (int oc = 0; oc < oc_n; ++oc) {
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
            uint4* dst = reinterpret_cast<uint4*>(orow + (own0 + oc0 + oc) * kChunk + hh * 32);
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
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bl.acc_free));
      t0 += g.ncols;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <int MODE, bool BF16>
cudaError_t launch_mode(const BwdParams& p_in, const BwdMaps& m, cudaStream_t st) {
  BwdParams p = p_in;
  constexpr int kMaxSmem = 232448;
  // Keep as many stationary operands resident as leave a ring of >= 3 stages
  // (>= 2 when nothing is resident).
  int n_res = (MODE == kDV) ? 1 : 2;
  int room = 0;
  for (; n_res >= 0; --n_res) {
    const Plan base = make_plan(p.n_chunks, 0, n_res, 1);
    room = kMaxSmem - 1024 - base.total;
    if (room / kChunkBytes >= 3) break;
  }
  if (n_res < 0) n_res = 0;
  // Two 16 KB tiles per ring slot when at least two such slots fit, else one.
  const int G = (room / (2 * kChunkBytes) >= 2) ? 2 : 1;
  int stages = room / (G * kChunkBytes);
  stages = min(stages, G == 2 ? 6 : 8);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  p.slot_chunks = G;
  const Plan plan = make_plan(p.n_chunks, stages, n_res, G);
  const int smem = plan.total + 1024;
  auto kern = bwd_main_kernel<MODE, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = (MODE == kDQ) ? dim3(p.q_tiles, p.Hq, p.B) : dim3(p.kv_tiles, p.Hkv, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  e = cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, m.dout, p, n_res);
  timing_mark(st);
  return e;
}

template <bool BF16>
cudaError_t launch_preprocess(const BwdParams& p, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Nq;
  timing_mark(st);
  bwd_preprocess_kernel<BF16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(p);
  timing_mark(st);
  return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_all(const BwdParams& p, const BwdMaps& m, cudaStream_t st) {
  cudaError_t e = launch_preprocess<BF16>(p, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_mode<kDV, BF16>(p, m, st)) != cudaSuccess) return e;
  if ((e = launch_mode<kDK, BF16>(p, m, st)) != cudaSuccess) return e;
  return launch_mode<kDQ, BF16>(p, m, st);
}

}  // namespace

cudaError_t launch_bwd(const BwdParams& p, const BwdMaps& m, bool bf16, cudaStream_t s) {
  if (bwd_xch_dkv_supported(p) && (bwd_dq_supported(p) || bwd_xch_dq_supported(p))) {
    // preprocess, the fused dK/dV kernel (two CTA pairs per key tile, or two
    // such clusters above D = 512), then dQ: one CTA pair per query tile up to
    // D = 512, two exchanging pairs above
    cudaError_t e = bf16 ? launch_preprocess<true>(p, s) : launch_preprocess<false>(p, s);
    if (e == cudaSuccess) e = launch_bwd_xch_dkv(p, m, bf16, s);
    if (e != cudaSuccess) return e;
    return bwd_dq_supported(p) ? launch_bwd_dq(p, m, bf16, s) : launch_bwd_xch_dq(p, m, bf16, s);
  }
  if (p.n_chunks <= 4) return bf16 ? launch_all<true>(p, m, s) : launch_all<false>(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace ffpa
