// Fused attention forward for D = 512 in which a CTA pair holds ALL of O for
// one 128-row query tile (tcgen05 cta_group::2 with M = 128).
//
// Same computation as fwd_main.cu: O = softmax(scale Q K^T + bias) V and the
// row logsumexp, keys in tiles of 128 with an online softmax.  Splitting O's
// 512 columns between two CTAs (or two pairs) makes each reduce S over the
// whole of D; here, as in the backward kernels (bwd_xch.cu, bwd_dq.cu), each SM of
// the pair holds 64 query rows of a 128 x 512 fp32 O across all 128 TMEM
// lanes (lane r: row r, the first N/2 columns of an accumulator; lane r + 64:
// the other N/2), so O takes 256 TMEM columns and S is computed once per key
// tile: about 4.6 Nq Nkv D executed per head (the residual term of P on part
// of the tiles included) instead of about 6.6.
//
// Per CTA c of the pair (query rows q0 + 64c .. q0 + 64c + 63):
//   * Q resident: columns 0..255 in TMEM as the A operand of the TS form (the
//     softmax threads load it from global memory; rows in both lane halves,
//     lanes r and r + 64, which the TS form of this MMA shape reads), columns
//     256..511 in shared memory (4 chunks of 64 rows x 64 columns, 32 KB).
//     The TMEM copy frees the shared memory for a second V slot;
//   * S_j = Q K_j^T: M = 128, N = 128, B split by N (this CTA loads keys
//     64c .. 64c + 63 of the key tile over all of D, 64 KB), into TMEM buffer
//     j mod 2 (64 columns: lane r keys 0..63 of row r, lane r + 64 keys
//     64..127);
//   * softmax by 128 threads, two per row (thread t: row t mod 64, key half
//     t / 64); the two swap their partial row maxima and sums through shared
//     memory at a named barrier of their two warps;
//   * P (and, on tiles that need it, its rounding residual) to shared memory as
//     the K-major A operand (64 rows x 128 keys, 16 KB each), in two buffers
//     used by alternate key tiles: an A operand in TMEM would have to sit in
//     both lane halves (lanes r and r + 64), which the score accumulator's
//     layout does not give, and one buffer made the softmax of tile j + 1
//     wait for P_j V;
//   * O += P V: two N = 256 MMAs per 16-key step (D columns 0..255 and
//     256..511), B split by N: this CTA loads 128 of each half's columns (32 KB
//     per half and key tile).  TMEM [128 h, 128 h + 128) holds half h: lane r
//     its columns 0..127, lane r + 64 its columns 128..255.
// Two threads of the first CTA issue the MMAs (one thread cannot issue pair
// MMAs and wait on barriers as fast as the tensor core runs them): thread A
// the S products from a ring of K tiles, thread B the P V products from a
// ring of V tiles; each ring has its own TMA producer.  Signals from the
// second CTA to the first: "S consumed" is a relaxed remote arrive (no data
// changes hands); "P written" needs a cluster-scope release, which costs the
// issuing thread about a thousand cycles, so the softmax warps arrive on a
// local barrier and an idle thread of that CTA (warp 2) forwards each phase.
//
// Warps: 0 K producer (and Q), 1 TMEM owner + MMA issuer A (first CTA), 2 MMA
// issuer B (first CTA) or the relay (second CTA), 3 V producer, 4-7 softmax /
// correction / epilogue.  Every wait is bounded (ptx.cuh).
#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace ffpa {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;            // rescale O only when the max grows by > 2^8
constexpr float kLoFrac = 1.0f / 64.0f;         // residual term of P only where a weight exceeds this share
constexpr int kHalfBytes = kChunkBytes / 2;     // 64 rows x 64 columns
constexpr int kPBytes = 2 * kHalfBytes;         // 64 rows x 128 keys, 16 KB
constexpr int kPBufBytes = 2 * kPBytes;         // P_hi and P_lo of one key tile
constexpr int kSlotBytes = 2 * kChunkBytes;     // 32 KB
constexpr int kKSlots = 2;

// Per head dimension D = 64 NC (NC = 5..16).
//
// O's columns: for D <= 512 one pair holds all of them; above, kNsplit pairs
// per query tile each hold a split of at most kOw columns (the last split may
// be narrower) and each reduces S over the whole of D.  A pair's P V product
// runs in up to two halves: its columns 0..255 (N = 256, or 128 when the split
// has at most 128 columns) and 256..256 + N1 - 1 (N1 = 128 or 256); V columns
// at or past D are zero-filled by TMA and the matching O columns not stored.
//
// TMEM (512 columns per SM): O in [0, kOTm) (half 0 from column 0, half 1 from
// column 128), the two 64-column score buffers, then Q's first kQtc chunks as
// the TS-form A operand (32 columns per chunk); Q's other chunks sit in shared
// memory.  Narrower O splits leave room for more of Q in TMEM, which is what
// lets shared memory hold the rest of Q next to the rings.  P is
// double-buffered where that shared memory allows (kNpb = 2).  Above D = 768
// the splits are 512 columns wide again (two pairs: S is computed twice, not
// three or four times) and the V ring has a single slot: the S product of
// such a key tile takes longer than the wait for V's second half.
template <int NC>
struct Shape {
  static_assert(NC >= 5 && NC <= 16, "D = 320 .. 1024");
  static constexpr int kD = 64 * NC;
  static constexpr int kOw = (NC <= 8 || NC >= 13) ? 512 : 384;  // widest O split
  static constexpr int kNsplit = (kD + kOw - 1) / kOw;
  static constexpr int kOTm = kOw / 2;                          // TMEM columns reserved for O
  // TMEM columns of O that a lane uses at most (rescale loop)
  static constexpr int kOCols = NC <= 8 ? 128 + (NC >= 7 ? 256 : 128) / 2 : kOTm;
  static_assert(kOTm <= 256, "O below the score buffers");
  static constexpr uint32_t kS0 = kOTm, kS1 = kOTm + 64, kQt = kOTm + 128;
  static constexpr int kQtc = (512 - static_cast<int>(kQt)) / 32 < NC ? (512 - static_cast<int>(kQt)) / 32 : NC;
  static constexpr int kQBytes = (NC - kQtc) * kHalfBytes;  // Q chunks kQtc..NC-1 in shared memory
  static constexpr int kNpb = NC - kQtc <= 4 ? 2 : 1;      // P buffers
  static constexpr int kKSlotsPerTile = (NC + 3) / 4;      // four K chunks (32 KB) per slot
  static constexpr int kVSlots = NC >= 13 ? 1 : 2;         // V ring slots (32 KB)
  // shared memory: Q | P buffers (P_hi, P_lo) | K ring | V ring | barriers | row-statistics exchange
  static constexpr int kPOff = kQBytes, kRingKOff = kPOff + kNpb * kPBufBytes;
  static constexpr int kRingVOff = kRingKOff + kKSlots * kSlotBytes;
  static constexpr int kMiscOff = kRingVOff + kVSlots * kSlotBytes;
  static constexpr int kSmemBytes = kMiscOff + 256 + 2 * 128 * 4 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "227 KB per CTA");
  static_assert(kOCols <= kOTm && kQtc >= 4, "TMEM layout");
};

struct Bars {
  int full_k, empty_k, full_v, empty_v, q_full, s_full, s_free, p_ready, p_local, pv_done, drain_a, drain_b, count;
};
// s_full, s_free: one per TMEM score buffer; p_ready, p_local, pv_done: one per P buffer
__host__ __device__ constexpr Bars bar_layout() {
  return Bars{0, 2, 4, 6, 8, 9, 11, 13, 15, 17, 19, 20, 21};
}
static_assert(bar_layout().count * 8 + 16 <= 256, "barrier area");

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
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Row r of a K-major, 128-byte-swizzled tile of 64 rows x 64 16-bit values:
// its eight 16-byte granules sit at r*128 + ((g ^ (r & 7)) << 4).
__device__ __forceinline__ void store_row64(uint32_t tile, int r, const uint32_t (&w)[32]) {
  const uint32_t row = tile + static_cast<uint32_t>(r) * 128u;
#pragma unroll
  for (int g = 0; g < 8; ++g)
    st_shared_v4(row + ((static_cast<uint32_t>(g) ^ static_cast<uint32_t>(r & 7)) << 4), w[4 * g], w[4 * g + 1],
                 w[4 * g + 2], w[4 * g + 3]);
}

// Named barrier of the two softmax warps that hold the two key halves of the
// same rows; returns the AND of their predicates (both then take the same branch).
__device__ __forceinline__ bool pair_bar_and(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

template <int NC, bool BF16, bool KSPLIT, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_fulld_kernel(const __grid_constant__ CUtensorMap map_qh, const __grid_constant__ CUtensorMap map_kh,
                     const __grid_constant__ CUtensorMap map_v, const __grid_constant__ FwdParams p) {
  using G = Shape<NC>;
  constexpr int kQBytes = G::kQBytes, kOCols = G::kOCols, kQtc = G::kQtc, kNpb = G::kNpb;
  constexpr uint32_t kS0 = G::kS0, kS1 = G::kS1, kQt = G::kQt;
  constexpr int kPOff = G::kPOff, kRingKOff = G::kRingKOff, kRingVOff = G::kRingVOff, kMiscOff = G::kMiscOff;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr Bars bl = bar_layout();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + bl.count);
  // lo_flag[j % kNpb] == j + 1: tile j carries the residual term of P.  The first
  // CTA's copy is read by thread B; the second CTA's softmax warps set their
  // own copy and its relay thread forwards it.
  volatile uint32_t* lo_flag = tmem_slot + 1;
  float* xmax = reinterpret_cast<float*>(smem + kMiscOff + 256);  // [128]: by TMEM lane
  float* xsum = xmax + 128;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t base = smem_u32(smem);
  const uint32_t q_sm = base, p_sm = base + kPOff;  // P buffer b: P_hi at p_sm + b kPBufBytes, P_lo 16 KB on
  const uint32_t ring_k = base + kRingKOff, ring_v = base + kRingVOff;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0 issues the pair's MMAs
  const int pair0 = static_cast<int>(blockIdx.x) >> 1;
  const int kvs = KSPLIT ? pair0 % p.kv_splits : 0;  // key split of this pair (KSPLIT: short query sets)
  const int pair = KSPLIT ? pair0 / p.kv_splits : pair0;
  const int split = pair % G::kNsplit;
  const int qt = p.q_tiles - 1 - pair / G::kNsplit;  // heavy causal tiles first
  const int q0 = qt * kTileRows;
  // this pair's O columns [o0, o0 + ow): halves of nv0 and nv1 64-column chunks per CTA
  const int o0 = split * G::kOw, ow = min(G::kOw, G::kD - o0);
  const int nv0 = ow >= 256 ? 2 : (ow + 127) / 128;
  const int nv1 = ow > 256 ? (ow - 256 + 127) / 128 : 0;
  const int nhalves = nv1 > 0 ? 2 : 1;
  const int h = blockIdx.y, b = blockIdx.z;
  const int kvh = h / p.group;
  const int kv_end = p.causal ? min(p.Nkv, q0 + kTileRows) : p.Nkv;
  // key tiles t0 .. t0 + ntiles - 1 (all of them without a key split)
  const int t0 = KSPLIT ? kvs * p.kv_split_tiles : 0;
  const int ntiles = KSPLIT ? max(0, min((kv_end + kTileRows - 1) / kTileRows - t0, p.kv_split_tiles))
                            : (kv_end + kTileRows - 1) / kTileRows;
  uint32_t* status = p.status;
  auto lead = [&](int i) { return rank == 0 ? bar(i) : mapa(bar(i), 0); };

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bl.full_k + i), 1);
      mbar_init(bar(bl.empty_k + i), 1);
      mbar_init(bar(bl.s_full + i), 1);
      mbar_init(bar(bl.s_free + i), 8);   // four softmax warps in each CTA
      mbar_init(bar(bl.p_ready + i), 5);  // this CTA's four softmax warps + the second CTA's relay
      mbar_init(bar(bl.p_local + i), 4);  // (second CTA) its four softmax warps
      mbar_init(bar(bl.pv_done + i), 1);
    }
    mbar_init(bar(bl.full_v), 1);
    mbar_init(bar(bl.empty_v), 1);
    mbar_init(bar(bl.full_v + 1), 1);
    mbar_init(bar(bl.empty_v + 1), 1);
    // Q ready: the producer's armed TMA bytes (chunks 4..NC-1) and the eight softmax
    // warps of the pair that wrote columns 0..255 into TMEM
    mbar_init(bar(bl.q_full), 1 + 8);
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
    // ------------------------------------------------------------ TMA producers (K and Q: warp 0, V: warp 3)
    // This CTA's slot s is free once the pair's MMAs reading it completed (the
    // first CTA's commit arrives on empty[s] here); the bytes are counted on
    // the first CTA's full[s], which that CTA arms for both halves.
    const bool is_k = warp == 0;
    const int full0 = is_k ? bl.full_k : bl.full_v, empty0 = is_k ? bl.empty_k : bl.empty_v;
    const uint32_t ring = is_k ? ring_k : ring_v;
    const uint32_t S = is_k ? kKSlots : G::kVSlots;
    if (is_k) {
      tma_prefetch_desc(&map_qh);
      tma_prefetch_desc(&map_kh);
      if (rank == 0) mbar_expect_tx(bar(bl.q_full), 2 * kQBytes);
      for (int c = kQtc; c < NC; ++c)
        tma_load_4d_pair(q_sm + (c - kQtc) * kHalfBytes, &map_qh, lead(bl.q_full), c * kChunk,
                         q0 + 64 * static_cast<int>(rank), h, b);
    } else {
      tma_prefetch_desc(&map_v);
    }
    bool ok = true;
    uint32_t it = 0;
    const int per_tile = is_k ? G::kKSlotsPerTile : nhalves;
    for (int n = 0; n < per_tile * ntiles && ok; ++n) {
      const uint32_t s = it % S, r = it / S;
      ++it;
      ok = mbar_wait<false>(bar(empty0 + s), (r & 1) ^ 1, status);
      if (!ok) break;
      const int j = n / per_tile, m = n % per_tile;
      // K: chunks 4m .. 4m + 3 (at most NC - 1) of this CTA's 64 keys of key
      // tile j; V: this CTA's share of O half m (one or two 64-column chunks)
      const int nk = min(4, NC - 4 * m), nv = m == 0 ? nv0 : nv1;
      if (rank == 0) mbar_expect_tx(bar(full0 + s), is_k ? 2 * nk * kHalfBytes : 2 * nv * kChunkBytes);
      const uint32_t dst = ring + s * kSlotBytes, fb = lead(full0 + s);
      if (is_k) {
        for (int i = 0; i < nk; ++i)
          tma_load_4d_pair(dst + i * kHalfBytes, &map_kh, fb, (4 * m + i) * kChunk,
                           (t0 + j) * kTileRows + 64 * static_cast<int>(rank), kvh, b);
      } else {
        for (int i = 0; i < nv; ++i)
          tma_load_4d_pair(dst + i * kChunkBytes, &map_v, fb, o0 + (4 * m + nv * static_cast<int>(rank) + i) * kChunk,
                           (t0 + j) * kTileRows, kvh, b);
      }
    }
    // the ring's last commits (they arrive on both CTAs) complete before exit
    for (uint32_t s = 0; s < S && s < it && ok; ++s) {
      const uint32_t last = s + ((it - 1 - s) / S) * S;
      mbar_wait<false>(bar(empty0 + s), (last / S) & 1, status);
    }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer A: S_j = Q K_j^T
    constexpr uint32_t idesc_s = idesc_f16(BF16, 128, 128, false, false);  // 128 rows x 128 keys
    const uint64_t dq = sdesc_sw128(q_sm, 16, 1024);                        // Q chunks (64 rows), K-major
    const uint64_t dk = sdesc_sw128(ring_k, 16, 1024);                      // K chunks (64 keys), K-major
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
      const uint32_t s_tm = tbase + ((j & 1) ? kS1 : kS0);
#pragma unroll
      for (int m = 0; m < G::kKSlotsPerTile; ++m) {
        const uint32_t s = it & 1;
        ok = mbar_wait<false>(bar(bl.full_k + s), (it >> 1) & 1, status);
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
              umma_ts_pair(s_tm, tbase + kQt + 32 * x + 8 * kk, sdesc_advance(bd, kk * 32), idesc_s, (x | kk) != 0);
          } else {  // Q from shared memory
            const uint64_t a = sdesc_advance(dq, (x - kQtc) * kHalfBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss_pair(s_tm, sdesc_advance(a, kk * 32), sdesc_advance(bd, kk * 32), idesc_s, 1u);
          }
        }
        umma_commit_pair(bar(bl.empty_k + s), 3);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.s_full + (j & 1)), 3);
    }
    umma_commit_pair(bar(bl.drain_a), 1);
    mbar_wait<false>(bar(bl.drain_a), 0, status);
  } else if (warp == 2 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------ MMA issuer B: O += P_j V_j
    constexpr uint32_t idesc_pv256 = idesc_f16(BF16, 128, 256, false, true);  // 128 rows x 256 O columns
    constexpr uint32_t idesc_pv128 = idesc_f16(BF16, 128, 128, false, true);  // 128 rows x 128 O columns
    const uint64_t dv = sdesc_sw128(ring_v, kChunkBytes, 1024);            // V chunk pairs, MN-major
    const uint64_t dp = sdesc_sw128(p_sm, 16, 1024);                       // P (64 rows x 128 keys), K-major
    bool ok = true;
    uint32_t it = 0;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int pb = j % kNpb;
      ok = mbar_wait<false>(bar(bl.p_ready + pb), (j / kNpb) & 1, status);
      if (!ok) break;
      tc_fence_after();
      const bool use_lo = lo_flag[pb] == static_cast<uint32_t>(j + 1);
      const uint64_t dphi = sdesc_advance(dp, pb * kPBufBytes), dplo = sdesc_advance(dphi, kPBytes);
      for (int hf = 0; hf < nhalves && ok; ++hf) {
        const uint32_t s = it % G::kVSlots;  // two slots (one per half of D), or one
        ok = mbar_wait<false>(bar(bl.full_v + s), (it / G::kVSlots) & 1, status);
        ++it;
        if (!ok) break;
        tc_fence_after();
        const uint64_t bd = sdesc_advance(dv, s * kSlotBytes);
        const uint32_t o_tm = tbase + 128 * hf;
        const uint32_t idesc_pv = (hf == 0 ? nv0 : nv1) == 2 ? idesc_pv256 : idesc_pv128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)  // 16-key steps: P subtile ks / 4, V rows 16 ks ..
          umma_ss_pair(o_tm, sdesc_advance(dphi, (ks >> 2) * kHalfBytes + (ks & 3) * 32),
                       sdesc_advance(bd, ks * 2048), idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        if (use_lo) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // the P_lo term
            umma_ss_pair(o_tm, sdesc_advance(dplo, (ks >> 2) * kHalfBytes + (ks & 3) * 32),
                         sdesc_advance(bd, ks * 2048), idesc_pv, 1u);
        }
        umma_commit_pair(bar(bl.empty_v + s), 3);
      }
      if (!ok) break;
      umma_commit_pair(bar(bl.pv_done + pb), 3);
    }
    umma_commit_pair(bar(bl.drain_b), 1);
    mbar_wait<false>(bar(bl.drain_b), 0, status);
  } else if (warp == 2 && lane == 0 && rank == 1) {
    // ------------------------------------------------------------ relay of this CTA's p_ready
    // The softmax warps of tile j + 2 wait for P_j V (pv_done of buffer j mod
    // 2), which needs this relay's arrive for tile j: a p_local barrier cannot
    // run two phases ahead.
    const uint32_t lo_flag_lead = mapa(smem_u32(const_cast<uint32_t*>(lo_flag)), 0);
    for (int j = 0; j < ntiles; ++j) {
      const int pb = j % kNpb;
      if (!mbar_wait<false>(bar(bl.p_local + pb), (j / kNpb) & 1, status)) break;
      if (lo_flag[pb] == static_cast<uint32_t>(j + 1)) st_cluster_u32(lo_flag_lead + 4 * pb, j + 1);
      mbar_arrive_remote(lead(bl.p_ready + pb));  // release.cluster: P and the flag are visible first
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / correction / epilogue
    const int t = tid - 128;      // TMEM lane
    const int r = t & 63;         // row within this CTA's 64
    const int kh = t >> 6;        // which 64 keys of each tile this thread scores
    const int row = q0 + 64 * static_cast<int>(rank) + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t nb = 1 + ((warp - 4) & 1);  // named barrier of warps w and w ^ 2 (lanes t and t ^ 64)
    const float* bias_row = nullptr;
    if (p.bias)
      bias_row = p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<int64_t>(min(row, p.Nq - 1)) * p.bias_sq;
    constexpr float kLog2e = 1.4426950408889634f;
    const uint32_t s_free_lead0 = lead(bl.s_free), s_free_lead1 = lead(bl.s_free + 1);
    const uint32_t p_ready_local = bar(rank == 0 ? bl.p_ready : bl.p_local);  // + 8 per P buffer
    {
      // Q columns 0 .. 64 kQtc - 1 of this thread's row into its TMEM lane: words of
      // two 16-bit values in memory order, the TS form's A layout (the threads of
      // lanes r and r + 64 write the same row)
      typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
      const uint4* qrow = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q) + b * p.q_sb + h * p.q_sh +
                                                         static_cast<int64_t>(min(row, p.Nq - 1)) * p.q_sn);
#pragma unroll
      for (int c = 0; c < kQtc; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 x = __ldg(qrow + 8 * c + g);
          w[4 * g] = x.x;
          w[4 * g + 1] = x.y;
          w[4 * g + 2] = x.z;
          w[4 * g + 3] = x.w;
        }
        tmem_st32(tbase + lane_off + kQt + 32 * c, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(bar(bl.q_full));
        else
          mbar_arrive_remote(lead(bl.q_full));
      }
    }
    bool ok = true;
    float m_used = -INFINITY, l_own = 0.f, l_sum = 0.f;  // l_sum: both halves of the row
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t s_col = (j & 1) ? kS1 : kS0;
      const int kv0 = (t0 + j) * kTileRows + 64 * kh;  // key of s[0]
      // this tile's bias row segment (256 bytes when contiguous) into L1 ahead of
      // the wait for S, so that the loads after it do not wait on L2
      if (bias_row && p.bias_vec) {
        prefetch_l1(bias_row + min(kv0, p.Nkv - 1));
        prefetch_l1(bias_row + min(kv0 + 32, p.Nkv - 1));
        prefetch_l1(bias_row + min(kv0 + 63, p.Nkv - 1));
      }
      // dropout: the keep bits of this thread's 64 keys, drawn while S is computed
      uint32_t keep_lo = 0, keep_hi = 0;
      if constexpr (DROP) {
        const DropKey dkey = {p.drop_seed_lo, p.drop_seed_hi, static_cast<uint32_t>(b * p.Hq + h), p.drop_off,
                              p.drop_t};
        keep64_row(dkey, kv0, row, keep_lo, keep_hi);
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
        // S_j is copied out: the buffer may take S_{j+2} ("consumed", no data hand-off)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          const uint32_t fr = (j & 1) ? s_free_lead1 : s_free_lead0;
          if (rank == 0)
            mbar_arrive(fr);
          else
            mbar_arrive_remote_relaxed(fr);
        }
      }
      const bool masked = (kv0 + 64 > p.Nkv) || (p.causal && kv0 + 63 > row);
      // Scores in the log2 domain: x = s scale log2e (+ bias log2e).  Without a
      // bias the scale is applied inside the exponent below (it is positive,
      // so the maximum of s gives the maximum of x).
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
      ok = pair_bar_and(nb, got);  // both warps of the pair see the same outcome
      if (!ok) break;
      const float m_tile = fmaxf(xmax[t], xmax[t ^ 64]);
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
      xsum[t] = l_own;
      pair_bar_and(nb, true);
      l_sum = xsum[t] + xsum[t ^ 64];
      // the residual term of P on this tile if some row's largest weight
      // exceeds 1/64 of its running sum (this tile included); the same in both
      // warps of the pair
      const bool warp_lo = __any_sync(0xffffffffu, ex2(m_tile - m_ref) > kLoFrac * l_sum);
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float p0 = s[2 * e], p1 = s[2 * e + 1];
        if constexpr (DROP) {  // dropped probabilities leave P V (the row sum above keeps them)
          const uint32_t kb = (e < 16 ? keep_lo : keep_hi) >> ((2 * e) & 31);
          p0 = (kb & 1u) ? p0 : 0.f;
          p1 = (kb & 2u) ? p1 : 0.f;
        }
        hi[e] = pack2<BF16>(p0, p1);
        if (warp_lo) {
          const float2 hv = unpack2<BF16>(hi[e]);
          lo[e] = pack2<BF16>(p0 - hv.x, p1 - hv.y);
        } else {
          lo[e] = 0u;
        }
      }
      const int pb = j % kNpb;
      if (j >= kNpb) {
        // P_{j-kNpb} V reads the P buffer this tile writes.  P_j V cannot have
        // completed, so the parity of that barrier is unambiguous.
        const bool done =
            __all_sync(0xffffffffu, mbar_wait<false>(bar(bl.pv_done + pb), ((j - kNpb) / kNpb) & 1, status));
        ok = pair_bar_and(nb, done);
        if (!ok) break;
      }
      const bool warp_rescale = __any_sync(0xffffffffu, rescale) && j >= 1;  // the same in both warps of the pair
      if (warp_rescale) {
        // the correction rewrites O: wait for P_{j-1} V (P_{j+1} V cannot have
        // completed, so the parity is unambiguous even where earlier tiles
        // skipped this wait)
        const bool done = __all_sync(
            0xffffffffu, mbar_wait<false>(bar(bl.pv_done + (j - 1) % kNpb), ((j - 1) / kNpb) & 1, status));
        ok = pair_bar_and(nb, done);
        if (!ok) break;
      }
      tc_fence_after();
      if (warp_rescale) {
        for (int c = 0; c < kOCols / 32; ++c) {  // this lane's O columns *= alpha
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
      // P of keys 64 kh .. 64 kh + 63 of row r: K-chunk kh of P buffer j mod kNpb
      const uint32_t pa = p_sm + pb * kPBufBytes;
      store_row64(pa + kh * kHalfBytes, r, hi);
      store_row64(pa + kPBytes + kh * kHalfBytes, r, lo);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (warp_lo) lo_flag[pb] = static_cast<uint32_t>(j + 1);
        mbar_arrive(p_ready_local + 8 * pb);  // release: P and the flag are visible first
      }
    }
    if (ok) {
      // ---------------------------------------------------------- epilogue
      // the last P V of each buffer (their commits also arrive on the second
      // CTA); a key split may have no key tile at all
      if (!KSPLIT || ntiles > 0)
        ok = __all_sync(0xffffffffu,
                        mbar_wait<false>(bar(bl.pv_done + (ntiles - 1) % kNpb), ((ntiles - 1) / kNpb) & 1, status));
      if (ok && kNpb == 2 && ntiles >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait<false>(bar(bl.pv_done + (ntiles & 1)), ((ntiles - 2) >> 1) & 1, status));
      if constexpr (KSPLIT) {
      if (ok) {
        // key split: the unnormalised partial O (fp32) and this split's (max,
        // sum) in the log2 domain, merged by the decode path's combine kernel
        tc_fence_after();
        const int prow_i = min(row, p.Nq - 1);
        float* prow = p.part_o + (((static_cast<int64_t>(b) * p.Hq + h) * p.Nq + prow_i) * p.kv_splits + kvs) * p.D;
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t v[32];
          if (ntiles > 0) {
            tmem_ld32(tbase + lane_off + c * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          // the O column of TMEM column 32 c of this lane, as in the epilogue below
          int d0;
          if (NC <= 8) {
            d0 = (c < 4 || NC >= 7) ? 256 * (c >> 2) + 128 * kh + 32 * (c & 3) : 256 + 64 * kh + 32 * (c - 4);
          } else if (c < 4) {
            d0 = c < 2 * nv0 ? o0 + 64 * nv0 * kh + 32 * c : NC * kChunk;
          } else {
            d0 = c - 4 < 2 * nv1 ? o0 + 256 + 64 * nv1 * kh + 32 * (c - 4) : NC * kChunk;
          }
          if (row < p.Nq && d0 < NC * kChunk) {
            float4* dst = reinterpret_cast<float4*>(prow + d0);
#pragma unroll
            for (int g = 0; g < 8; ++g)
              dst[g] = make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                   __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
          }
        }
        if (kh == 0 && split == 0 && row < p.Nq) {
          float* ml = p.part_ml + (((static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row) * p.kv_splits + kvs) * 2;
          ml[0] = ntiles > 0 ? m_used : -INFINITY;
          ml[1] = l_sum;
        }
      }
      } else {
      if (ok) {
        tc_fence_after();
        // dropout: kept probabilities carry 1 / (1 - p)
        const float inv_l = l_sum > 0.f ? (DROP ? p.drop_scale : 1.f) / l_sum : 0.f;
        typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
        T* orow = reinterpret_cast<T*>(p.out) + b * p.o_sb + h * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + c * 32, v);
          tmem_ld_wait();
          if (row < p.Nq) {
            // TMEM column 32 c + i of lane 64 kh + r is O column o0 + (N0 / 2) kh
            // + 32 c + i (half 0, c < N0 / 64) or o0 + 256 + (N1 / 2) kh + 32 (c - 4)
            // + i (half 1, c >= 4), with N_h = 128 nv_h
            int d0;
            if constexpr (NC <= 8) {
              constexpr bool kN1Wide = NC >= 7;                 // N1 = 256
              constexpr bool kPadded = NC == 5 || NC == 7;      // the last O columns are padding
              d0 = (c < 4 || kN1Wide) ? 256 * (c >> 2) + 128 * kh + 32 * (c & 3) : 256 + 64 * kh + 32 * (c - 4);
              if (kPadded && d0 >= NC * kChunk) continue;  // zero-filled V columns past D
            } else {
              if (c < 4) {
                if (c >= 2 * nv0) continue;
                d0 = o0 + 64 * nv0 * kh + 32 * c;
              } else {
                if (c - 4 >= 2 * nv1) continue;
                d0 = o0 + 256 + 64 * nv1 * kh + 32 * (c - 4);
              }
              if (d0 >= NC * kChunk) continue;
            }
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
        if (kh == 0 && split == 0 && p.lse && row < p.Nq) {
          constexpr float kLn2 = 0.6931471805599453f;
          p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] =
              l_sum > 0.f ? (m_used + __log2f(l_sum)) * kLn2 : -INFINITY;
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
  p.stages = kKSlots + Shape<NC>::kVSlots;
  p.slot_chunks = 2;
  // key splits and dropout are not combined (the host takes no key split with dropout)
  auto kern = p.part_o ? fwd_fulld_kernel<NC, BF16, true, false>
                       : (p.dropout ? fwd_fulld_kernel<NC, BF16, false, true> : fwd_fulld_kernel<NC, BF16, false, false>);
  constexpr int kNsplit = Shape<NC>::kNsplit;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.q_tiles * kNsplit * (p.part_o ? p.kv_splits : 1), p.Hq, p.B);  // (pair rank, key split, O split, query tile)
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

template <int NC>
cudaError_t launch_nc(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  return bf16 ? launch_impl<NC, true>(p, m, s) : launch_impl<NC, false>(p, m, s);
}

}  // namespace

bool fwd_fulld_supported(const FwdParams& p) { return p.n_chunks >= 5 && p.n_chunks <= 16; }

// Key splits for short query sets: when the pairs of a launch would not fill
// one wave of pair slots, split the keys so that about one wave runs, each
// split at least two key tiles long.  Returns the split count (1: none) and
// the key tiles per split.
int fwd_fulld_kv_splits(const FwdParams& p, int sms, int* tiles_per_split) {
  if (p.dropout) {  // no key-split form of the dropout kernel
    *tiles_per_split = (p.Nkv + kTileRows - 1) / kTileRows;
    return 1;
  }
  int nsplit = 1;
  switch (p.n_chunks) {
    case 9: nsplit = Shape<9>::kNsplit; break;
    case 10: nsplit = Shape<10>::kNsplit; break;
    case 11: nsplit = Shape<11>::kNsplit; break;
    case 12: nsplit = Shape<12>::kNsplit; break;
    case 13: nsplit = Shape<13>::kNsplit; break;
    case 14: nsplit = Shape<14>::kNsplit; break;
    case 15: nsplit = Shape<15>::kNsplit; break;
    case 16: nsplit = Shape<16>::kNsplit; break;
    default: nsplit = 1;
  }
  const int64_t pairs = static_cast<int64_t>(p.q_tiles) * nsplit * p.Hq * p.B;
  const int kv_tiles = (p.Nkv + kTileRows - 1) / kTileRows;
  const int64_t slots = sms / 2;
  *tiles_per_split = kv_tiles;
  if (pairs * 2 > slots || kv_tiles < 4) return 1;  // half a wave or more: no split
  const int want = static_cast<int>(std::min<int64_t>(slots / pairs, kv_tiles / 2));
  if (want < 2) return 1;
  const int per = (kv_tiles + want - 1) / want;
  *tiles_per_split = per;
  return (kv_tiles + per - 1) / per;
}

cudaError_t launch_fwd_fulld(const FwdParams& p, const FwdMaps& m, bool bf16, cudaStream_t s) {
  switch (p.n_chunks) {
    case 5: return launch_nc<5>(p, m, bf16, s);
    case 6: return launch_nc<6>(p, m, bf16, s);
    case 7: return launch_nc<7>(p, m, bf16, s);
    case 8: return launch_nc<8>(p, m, bf16, s);
    case 9: return launch_nc<9>(p, m, bf16, s);
    case 10: return launch_nc<10>(p, m, bf16, s);
    case 11: return launch_nc<11>(p, m, bf16, s);
    case 12: return launch_nc<12>(p, m, bf16, s);
    case 13: return launch_nc<13>(p, m, bf16, s);
    case 14: return launch_nc<14>(p, m, bf16, s);
    case 15: return launch_nc<15>(p, m, bf16, s);
    default: return launch_nc<16>(p, m, bf16, s);
  }
}

}  // namespace ffpa
