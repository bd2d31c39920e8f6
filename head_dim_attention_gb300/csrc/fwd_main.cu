// Fused attention forward on sm_103a: the one-CTA kernel for D <= 256 and the
// forward's dispatch.
//
// O = softmax(scale * Q K^T + bias) V and lse (natural log), the plain
// definition in the attention-kernel-profiler design notes (generate_docs.py,
// DESIGN section 3, "naive_math"), computed without materialising S: the keys
// stream in tiles of 128 with an online softmax (running max and sum, lazy
// rescale of O).
//
// This kernel covers D <= 256, where one CTA holds all of O (at most 256 fp32
// TMEM columns) next to two 128-column score buffers.  Every larger head
// dimension (320 .. 1024) goes to the CTA-pair kernel of fwd_fulld.cu, which
// launch_fwd_main below hands it to: there two SMs hold O's columns for one
// 128-row query tile across all 128 TMEM lanes (the FFPA pages' fine tiling
// along D, FFPA-Attn Performance Benchmarks page, "Why the Trends Look Like
// This", applied to TMEM instead of registers and shared memory).
//
// Warp roles (256 threads): warps 0, 2 and 3 = TMA producers, warp 1 = TMEM
// owner and MMA issuer, warps 4-7 = softmax / correction / epilogue (one query row per
// thread; warp 4+w reads TMEM lanes 32w..32w+31).
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 256;
constexpr int kProducers = 3;  // warps 0, 2 and 3
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kS0 = 256, kS1 = 384;  // TMEM columns of the two S/P buffers
constexpr int kMaxChunks = 4;             // D <= 256: O in TMEM columns [0, 256)
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the max grows by > 2^8
// A key tile feeds P to P V as two 16-bit terms only when some row of it holds
// a probability above this fraction of the row's running sum (see below).
constexpr float kLoFrac = 1.0f / 64.0f;

struct Bars {
  // indices into the barrier array
  int full, empty, q_full, s_full, p_ready, o_ready, drain, count;
};
__host__ __device__ inline Bars bar_layout(int stages) {
  Bars b;
  b.full = 0;
  b.empty = stages;
  b.q_full = 2 * stages;
  b.s_full = b.q_full + 1;   // 2
  b.p_ready = b.s_full + 2;  // 2
  b.o_ready = b.p_ready + 2;
  b.drain = b.o_ready + 1;
  b.count = b.drain + 1;
  return b;
}

// shared memory: Q (all chunks, resident) | ring | barriers + TMEM slot
struct SmemPlan {
  int q_off, ring_off, bar_off, total;
};
__host__ __device__ inline SmemPlan smem_plan(int n_chunks, int stages, int slot_chunks) {
  SmemPlan s;
  s.q_off = 0;
  s.ring_off = n_chunks * kChunkBytes;
  s.bar_off = s.ring_off + stages * slot_chunks * kChunkBytes;
  s.total = s.bar_off + 1024;
  return s;
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
    fwd_main_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const __grid_constant__ FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int stages = p.stages;
  const int G = p.slot_chunks;                  // chunk tiles per ring slot
  const uint32_t slot_bytes = G * kChunkBytes;
  const SmemPlan plan = smem_plan(p.n_chunks, stages, G);
  const Bars bl = bar_layout(stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  // lo_flag[t & 1] == t + 1: tile t carries the residual term of P (written by
  // the softmax warps before they arrive on p_ready, read by the MMA thread after)
  volatile uint32_t* lo_flag = tmem_slot + 1;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t s_base = smem_u32(smem);
  const uint32_t q_sm = s_base + plan.q_off, ring_sm = s_base + plan.ring_off;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = p.q_tiles - 1 - static_cast<int>(blockIdx.x);  // heavy causal tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / p.group;
  const int q0 = qt * kTileRows;
  const int n = p.n_chunks;  // chunks of D: S reduces over them, O holds them
  const int kv_end = p.causal ? min(p.Nkv, q0 + kTileRows) : p.Nkv;
  const int ntiles = (kv_end + kTileRows - 1) / kTileRows;
  uint32_t* status = p.status;

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar(bl.full + i), 1);
      mbar_init(bar(bl.empty + i), 1);
    }
    mbar_init(bar(bl.q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.s_full + i), 1);
      mbar_init(bar(bl.p_ready + i), 4);
    }
    mbar_init(bar(bl.o_ready), 1);
    mbar_init(bar(bl.drain), 1);
    lo_flag[0] = 0;
    lo_flag[1] = 0;
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
    // nprod-th load of the sequence and waits only for its own slot to be
    // released. Arming a barrier and issuing a TMA load blocks the issuing
    // thread for ~500 cycles, so one thread alone cannot keep the ring full.
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
      if (pi == 0) {
        mbar_expect_tx(bar(bl.q_full), n * kChunkBytes);
        for (int c = 0; c < n; ++c) tma_load_4d(q_sm + c * kChunkBytes, &map_q, bar(bl.q_full), c * kChunk, q0, h, b);
      }
      bool ok = true;
      uint32_t it = 0;
      // One ring slot takes `cn` (<= G) consecutive 64-column chunk tiles under
      // a single barrier phase.  Each phase of a slot (arm, land, wait, release)
      // costs the SM a few hundred cycles whatever its size, so two 16 KB tiles
      // per phase move nearly twice the bytes of one.
      auto load = [&](const CUtensorMap* m, int c0, int cn, int row) {
        if (ok && static_cast<int>(it % nprod) == pi) {
          const uint32_t s = it % stages, r = it / stages;
          ok = mbar_wait(bar(bl.empty + s), (r & 1) ^ 1, status);
          if (ok) {
            mbar_expect_tx(bar(bl.full + s), cn * kChunkBytes);
            for (int i = 0; i < cn; ++i)
              tma_load_4d(ring_sm + s * slot_bytes + i * kChunkBytes, m, bar(bl.full + s), (c0 + i) * kChunk, row,
                          kvh, b);
          }
        }
        ++it;
      };
      // K of tile j, then V of tile j - 1: the order the MMA thread uses them
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles)
          for (int c = 0; c < n; c += G) load(&map_k, c, min(G, n - c), j * kTileRows);
        if (j >= 1)
          for (int c = 0; c < n; c += G) load(&map_v, c, min(G, n - c), (j - 1) * kTileRows);
      }
      // Drain: wait for the last release of each ring slot whose last load was
      // ours. The MMA warp's commit arrives on empty[s] only when the MMAs
      // reading the slot are done, and commit arrivals are not ordered with
      // respect to one another, so one still in flight at exit would land in
      // the next CTA's shared memory.
      for (uint32_t s = 0; s < static_cast<uint32_t>(stages) && s < it; ++s) {
        const uint32_t last = s + ((it - 1 - s) / stages) * stages;
        if (static_cast<int>(last % nprod) == pi) mbar_wait(bar(bl.empty + s), (last / stages) & 1, status);
      }
      if (pi == 0) mbar_wait(bar(bl.q_full), 0, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are formed once and advanced by constants: building them per
    // MMA made the issuing thread, not the tensor pipe, the bottleneck.
    if (lane == 0) {
      const uint32_t idesc_s128 = idesc_f16(BF16, 128, 128, false, false);  // a whole key tile
      const uint32_t idesc_pv = idesc_f16(BF16, 128, 64, false, true);      // one V chunk
      const uint32_t idesc_pv2 = idesc_f16(BF16, 128, 128, false, true);    // two V chunks in adjacent slots
      const uint64_t dq = sdesc_sw128(q_sm, 16, 1024);                      // Q chunks, K-major
      const uint64_t dk = sdesc_sw128(ring_sm, 16, 1024);                   // ring tiles as K-major operands
      const uint64_t dv = sdesc_sw128(ring_sm, kChunkBytes, 1024);          // ring tiles as MN-major operands
      bool ok = mbar_wait(bar(bl.q_full), 0, status);
      tc_fence_after();
      uint32_t it = 0;
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles) {
          // S_t lands in the buffer that held P_{t-2}, the A operand of the
          // P_{t-2} V MMA; tcgen05.mma does not order a later MMA's write of D
          // after an earlier MMA's read of A from TMEM, so S_t is issued once
          // that MMA has completed.  S is issued whole (N=128): splitting it
          // into N=64 halves to start earlier measured slower.
          const int t = j;
          const uint32_t s_tm = tbase + ((t & 1) ? kS1 : kS0);
          if (j >= 2) {
            ok = mbar_wait(bar(bl.o_ready), (t - 2) & 1, status);
            if (!ok) break;
            tc_fence_after();
          }
          for (int c = 0; c < n && ok; c += G) {
            const uint32_t s = it % stages;
            ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            const int cn = min(G, n - c);
            for (int i = 0; i < cn; ++i) {
              const uint64_t a = sdesc_advance(dq, (c + i) * kChunkBytes);
              const uint64_t bd = sdesc_advance(dk, s * slot_bytes + i * kChunkBytes);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss(s_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_s128,
                        ((c + i) | kk) != 0);
            }
            umma_commit(bar(bl.empty + s));
            ++it;
          }
          if (!ok) break;
          umma_commit(bar(bl.s_full + (t & 1)));
        }
        if (j >= 1 && ok) {
          const int t = j - 1;
          ok = mbar_wait(bar(bl.p_ready + (t & 1)), (t >> 1) & 1, status);
          if (!ok) break;
          tc_fence_after();
          const bool use_lo = lo_flag[t & 1] == static_cast<uint32_t>(t + 1);
          const uint32_t p_tm = tbase + ((t & 1) ? kS1 : kS0);
          // O[:, c..] += P V[:, c..]: two chunks per MMA (N=128) when they share
          // a ring slot, or (one chunk per slot) sit in adjacent slots
          for (int c = 0; c < n && ok;) {
            const uint32_t s = it % stages;
            if (G == 2) {
              ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
              if (!ok) break;
              tc_fence_after();
              const uint64_t bd = sdesc_advance(dv, s * slot_bytes);
              const uint32_t acc0 = (j - 1 > 0) ? 1u : 0u;
              const uint32_t idesc = (c + 1 < n) ? idesc_pv2 : idesc_pv;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + c * kChunk, p_tm + kk * 8, sdesc_advance(bd, kk * 2048), idesc, acc0 | (kk > 0));
              if (use_lo) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // the P_lo term
                  umma_ts(tbase + c * kChunk, p_tm + 64 + kk * 8, sdesc_advance(bd, kk * 2048), idesc, 1u);
              }
              umma_commit(bar(bl.empty + s));
              it += 1;
              c += 2;
              continue;
            }
            const bool two = (c + 1 < n) && (s + 1 < static_cast<uint32_t>(stages));
            ok = mbar_wait(bar(bl.full + s), (it / stages) & 1, status);
            if (ok && two) ok = mbar_wait(bar(bl.full + s + 1), ((it + 1) / stages) & 1, status);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bd = sdesc_advance(dv, s * kChunkBytes);
            const uint32_t acc0 = (j - 1 > 0) ? 1u : 0u;
            if (two) {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + c * kChunk, p_tm + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv2, acc0 | (kk > 0));
              if (use_lo) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // the P_lo term
                  umma_ts(tbase + c * kChunk, p_tm + 64 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv2, 1u);
              }
              umma_commit(bar(bl.empty + s));
              umma_commit(bar(bl.empty + s + 1));
              it += 2;
              c += 2;
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_ts(tbase + c * kChunk, p_tm + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv, acc0 | (kk > 0));
              if (use_lo) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)  // the P_lo term
                  umma_ts(tbase + c * kChunk, p_tm + 64 + kk * 8, sdesc_advance(bd, kk * 2048), idesc_pv, 1u);
              }
              umma_commit(bar(bl.empty + s));
              it += 1;
              c += 1;
            }
          }
          umma_commit(bar(bl.o_ready));
        }
      }
      umma_commit(bar(bl.drain));
      mbar_wait(bar(bl.drain), 0, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / correction / epilogue
    const int r = tid - 128;  // query row within the tile == TMEM lane
    const int row = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const float* bias_row = nullptr;
    if (p.bias)
      bias_row = p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(min(row, p.Nq - 1)) * p.bias_sq;
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;
    float m_used = -INFINITY, l_sum = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      const int t = j;
      const uint32_t s_col = (t & 1) ? kS1 : kS0;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.s_full + (t & 1)), (t >> 1) & 1, status));
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + s_col + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      // scale (log2 domain), bias, masks
      const int kv0 = j * kTileRows;
      const bool masked = (kv0 + kTileRows > p.Nkv) || (p.causal && kv0 + kTileRows - 1 > row);
      const float c_scale = p.scale_log2;
      if (bias_row) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          s[i] = fmaf(__ldg(bias_row + static_cast<int64_t>(kv0 + min(i, p.Nkv - 1 - kv0)) * p.bias_sk), kLog2e,
                      s[i] * c_scale);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] *= c_scale;
      }
      if (masked) {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int kv = kv0 + i;
          if (kv >= p.Nkv || (p.causal && kv > row)) s[i] = -INFINITY;
        }
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 128; ++i) mx[i & 3] = fmaxf(mx[i & 3], s[i]);
      const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
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
      for (int i = 0; i < 128; ++i) {
        s[i] = ex2(s[i] - m_ref);  // P, in place
        ls[i & 3] += s[i];
      }
      l_sum = l_sum * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      // Rounding P to 16 bits perturbs each weight by up to 2^-8 of itself
      // (bf16).  That matters only for rows where a few keys carry much of
      // the weight (outputs that are sums of a few nearly cancelling V rows);
      // in a row whose weight is spread, the rounding errors of many small
      // terms average out far below the tolerance.  So the residual term is
      // fed only when this tile's largest probability exceeds kLoFrac of the
      // row's running sum (the final sum is larger still).
      const bool warp_lo = __any_sync(0xffffffffu, ex2(m_tile - m_ref) > kLoFrac * l_sum);
      if (j >= 1) {
        // Wait for the previous P V MMA before touching TMEM again: storing P
        // while that MMA ran gave wrong O on GB300 (found by testing, single-
        // CTA configuration), and the O correction below needs it anyway.
        // The MMA is short, so this wait is normally already satisfied.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.o_ready), (t - 1) & 1, status));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale) && j >= 1) {
        // correction: O of this row *= alpha
        for (int c = 0; c < n; ++c) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            const uint32_t a = tbase + lane_off + c * kChunk + hh * 32;
            tmem_ld32(a, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(a, v);
          }
        }
      }
      // P goes to TMEM as two terms of the input type, P = P_hi + P_lo with
      // P_lo the rounding residual of P_hi (columns 0..63 and 64..127 of the
      // score buffer); the P V product sums both, so the 16-bit operand costs
      // about 2^-17 of P instead of 2^-8 (bf16).  A warp whose rows do not
      // need the residual stores zeros there, in case another warp's rows
      // make the MMA thread issue the residual product for the whole tile.
      if (warp_lo) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = s[32 * g + 2 * e], p1 = s[32 * g + 2 * e + 1];
            hi[e] = pack2<BF16>(p0, p1);
            const float2 h = unpack2<BF16>(hi[e]);
            lo[e] = pack2<BF16>(p0 - h.x, p1 - h.y);
          }
          tmem_st16(tbase + lane_off + s_col + 16 * g, hi);
          tmem_st16(tbase + lane_off + s_col + 64 + 16 * g, lo);
        }
      } else {
        uint32_t zero[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) zero[e] = 0u;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t hi[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) hi[e] = pack2<BF16>(s[32 * g + 2 * e], s[32 * g + 2 * e + 1]);
          tmem_st16(tbase + lane_off + s_col + 16 * g, hi);
          tmem_st16(tbase + lane_off + s_col + 64 + 16 * g, zero);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (warp_lo) lo_flag[t & 1] = static_cast<uint32_t>(t + 1);
        mbar_arrive(bar(bl.p_ready + (t & 1)));  // release: the flag store is visible first
      }
    }
    // ---------------------------------------------------------- epilogue
    const int t_last = ntiles - 1;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(bl.o_ready), t_last & 1, status));
    if (ok) {
      tc_fence_after();
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
      T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
      for (int c = 0; c < n; ++c) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + c * kChunk + hh * 32, v);
          tmem_ld_wait();
          if (row < p.Nq) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * kChunk + hh * 32);
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
      if (p.lse && row < p.Nq) {
        constexpr float kLn2 = 0.6931471805599453f;
        p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] =
            l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

template <bool BF16>
cudaError_t launch_impl(const FwdParams& p_in, const FwdMaps& m, cudaStream_t st) {
  FwdParams p = p_in;
  constexpr int kMaxSmem = 232448;  // 227 KB opt-in per block
  const SmemPlan base = smem_plan(p.n_chunks, 0, 1);
  const int room = kMaxSmem - 1024 - base.total;
  // Two chunk tiles per ring slot when at least two such slots fit, else one.
  int G = (room / (2 * kChunkBytes) >= 2) ? 2 : 1;
  int stages = room / (G * kChunkBytes);
  stages = min(stages, G == 2 ? 6 : 8);
  if (stages < 2) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  p.slot_chunks = G;
  const SmemPlan plan = smem_plan(p.n_chunks, stages, G);
  const int smem = plan.total + 1024;  // + alignment slack
  auto kern = fwd_main_kernel<BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.q_tiles, p.Hq, p.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  timing_mark(st);
  e = cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, p);
  timing_mark(st);
  return e;
}

}  // namespace

cudaError_t launch_fwd_main(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  if (fwd_xch_supported(p)) return launch_fwd_xch(p, m, bf16, s);      // D = 704 .. 1024
  if (fwd_fulld_supported(p)) return launch_fwd_fulld(p, m, bf16, s);  // D = 320 .. 1024
  if (p.n_chunks > kMaxChunks) return cudaErrorInvalidValue;
  return bf16 ? launch_impl<true>(p, m, s) : launch_impl<false>(p, m, s);
}

}  // namespace ffpa
