// argus_window_prefill_attn: attention of a query chunk against one window of
// cached keys, folded into an fp32 accumulator by log2-sum-exp.
//
// "feat(kvcache): host-RAM KV tier for sparse-attention models", comment on
// "--kv-placement host": when the in-place reads of a prefill's rows add up to
// more bytes than the cache holds, the cached pages are staged into a 131,072-token device window,
// attended per window, and the windows folded by their log2-sum-exp into a
// float32 accumulator allocated up front (fold_attention_pass).
//
// GB300 design: this is the one dense contraction of the library, so it runs
// on the 5th-generation tensor cores.
//  * A CTA owns 128 query rows of one KV head: the G query heads sharing the KV
//    head are stacked along M, so every K/V tile loaded is used by all of them.
//  * TMA (cp.async.bulk.tensor, 128-byte swizzle) streams the Q tile once and
//    128-key K/V tiles through a two-stage ring.
//  * One elected thread issues tcgen05.mma: S = Q K^T (M=128, N=128, K=16 steps)
//    into one of two TMEM score buffers while the softmax warps work on the
//    other, then O += P V with P read straight from TMEM (it overwrites the
//    consumed scores, as a bf16 hi + lo pair) and V from shared memory
//    (MN-major operand).
//  * Four softmax warps own one query row per thread (TMEM lane = row): scores
//    are read with tcgen05.ld, the running max is only moved when it grows by
//    more than 2^8 (the exact result does not depend on the reference), and the
//    rare rescale of O goes through TMEM.
//  * The epilogue normalises O, forms lse2 = m + log2(l) and folds the window
//    into the caller's fp32 accumulator.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace argus {
namespace prefill {

constexpr int kBM = 128;          // query rows per CTA (TMEM lanes)
constexpr int kBN = 128;          // keys per block
constexpr int kStages = 3;        // K/V ring depth
constexpr int kGroupWarps = 4;    // one softmax warpgroup: a thread per row
constexpr int kSoftmaxWarps = 2 * kGroupWarps;   // two groups take alternate key blocks
constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
constexpr int kHalf = kBM * 64 * 2;   // 16 KB: 128 rows x 64 dims, one 128-byte swizzle column
constexpr int kTmemCols = 512;        // S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D)
constexpr float kRescaleThreshold = 8.f;

// Shared memory map of head_dim D (offsets from a 1024-byte aligned base): a
// 128-row bf16 / fp16 tile is D / 64 swizzled 16 KB halves of 64 dims each.
template <int D>
struct Smem {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kTile;
  static constexpr int kOffV = kOffK + kStages * kTile;
  static constexpr int kOffBar = kOffV + kStages * kTile;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], s_free[2], o_done[2]
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffML = kOffMisc + 64;                 // group 1's (m, l) per row
  static constexpr int kBytes = kOffML + kBM * 8 + 1024;       // + alignment slack
};

struct PParams {
  int G, n_q, n_tiles;              // tiles per KV head = ceil(G * n_q / 128)
  long long rows_h;                 // query rows per KV head = G * n_q (its G heads stacked)
  long long win_len, win_pos0, q_pos0;
  float scale_log2;
  float* acc_o;
  float* acc_lse2;
  int fold;
  int nsplit;                       // key ranges per tile (grid.z)
  float* ws_o;                      // nsplit > 1: partial o [tile][split][128][D], normalised
  float* ws_lse;                    //             and its lse2 [tile][split][128]
  const uint32_t* vmax_bits;        // fp16 P.V: bits of max |v| over the window
  // fp16 Q.K^T (staged paged windows): K scaled by 2^-ek from max |k| (bits at
  // kmax_bits), query row r scaled by 1 / qfac[r]; score = S' * qfac[r] * 2^ek
  const uint32_t* kmax_bits;
  const float* qfac;
};

// fp16 copies (V for fp16 P.V; K and V of a staged paged window) are scaled by
// 2^-e with e chosen from the largest magnitude m of the copied values so that
// m * 2^-e lies in [2^14, 2^15): nothing overflows fp16 and small values keep
// their precision.  The result is multiplied back by 2^e.  Every thread derives
// e from the same max word.  m = 0 (or not finite) gives e = 0.
__device__ __forceinline__ int f16_exponent(uint32_t max_bits) {
  const float m = __uint_as_float(max_bits);
  if (!(m > 0.f) || !(m < 3.0e38f)) return 0;
  int k = 0;
  frexpf(m, &k);                                     // 2^(k-1) <= m < 2^k
  return k - 15;
}

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor, 128-byte swizzle (sm_100 layout code 2, version 1)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16 -> f32, M = 128, N = n; operand type
// 1 = bf16 (both operands), 0 = fp16 (both operands)
__host__ __device__ constexpr uint32_t idesc_f16kind(bool bf16, bool b_mn_major, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- kernel
__device__ __forceinline__ void group_bar(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kSoftmaxWarps * 32) : "memory");
}

// MODE 0: Q.K^T in bf16, P.V in bf16 with P split into hi + lo parts (two MMAs).
// MODE 1: Q.K^T in bf16, P.V in fp16 (P scaled by 2^7, V the scaled fp16 copy),
//         one MMA per key step.
// MODE 2: both in fp16 over a staged window: fp16 K and V copies scaled by
//         powers of two and an fp16 query scaled per row (score scale per row).
template <int MODE, int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PParams p) {
  using SM = Smem<D>;
  constexpr int kTile = SM::kTile;
  constexpr bool F16P = MODE >= 1;
  constexpr bool F16QK = MODE == 2;
  constexpr float kPBias = F16P ? 7.f : 0.f;   // fp16 P is stored as P * 2^kPBias
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* s_free = p_full + 2;
  uint64_t* o_done = s_free + 2;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + SM::kOffMisc);  // [0] tmem base, [1] error
  float2* ml1 = reinterpret_cast<float2*>(smem + SM::kOffML);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, h = blockIdx.y, split = blockIdx.z;
  // The G query heads of KV head h are stacked: row lin of the head's rows_h
  // rows is query index lin % n_q of query head h * G + lin / n_q, and Q / the
  // accumulator row h * rows_h + lin.  A tile may straddle two query heads; its
  // rows past rows_h (last tile) are computed on whatever the load gave and
  // never written.
  const long long lin0 = (long long)tile * kBM;
  const long long row0 = (long long)h * p.rows_h + lin0;                      // first row of [Hq*n_q]
  const long long lin_last = min(lin0 + kBM - 1, p.rows_h - 1);
  const long long qi_max = (lin0 / p.n_q != lin_last / p.n_q) ? p.n_q - 1 : lin_last % p.n_q;
  // keys j < n_keys can be visible to some row of the tile
  const long long last_visible = p.q_pos0 + qi_max - p.win_pos0;
  long long n_keys = last_visible + 1;
  if (n_keys < 0) n_keys = 0;
  if (n_keys > p.win_len) n_keys = p.win_len;
  const int nb_tile = (int)((n_keys + kBN - 1) / kBN);
  // this CTA's key blocks: [jb, jb + nb) of the tile's nb_tile, balanced over the splits
  const int jb = (int)((long long)split * nb_tile / p.nsplit);
  const int nb = (int)((long long)(split + 1) * nb_tile / p.nsplit) - jb;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], kGroupWarps);   // one arrival per softmax warp
      mbar_init(&s_free[b], 1);
      mbar_init(&o_done[b], 1);
    }
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kSoftmaxWarps + 1) {  // the MMA warp owns the TMEM allocation
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((const void*)&misc[0])),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // TMEM columns of score buffer b and O accumulator b (arithmetic, not a
  // table: a runtime index into an array would put it in local memory)
  auto tS = [tmem](int b) { return tmem + 128u * (uint32_t)b; };
  auto tO = [tmem](int b) { return tmem + 256u + 128u * (uint32_t)b; };

  if (warp == kSoftmaxWarps) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0 && nb > 0) {
      mbar_arrive_expect_tx(q_full, kTile);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(smem + SM::kOffQ + hf * kHalf, &tmQ, 64 * hf, (int)row0, q_full);
      for (int i = 0; i < nb; ++i) {
        const int st = i % kStages;
        const int y = (jb + i) * kBN;
        if (i >= kStages && !mbar_wait(&kv_empty[st], ((i / kStages) - 1) & 1, &misc[1])) {
          misc[1] = 1;
          break;
        }
        mbar_arrive_expect_tx(&kv_full[st], 2 * kTile);
        uint8_t* kd = smem + SM::kOffK + st * kTile;
        uint8_t* vd = smem + SM::kOffV + st * kTile;
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_3d(kd + hf * kHalf, &tmK, 64 * hf, y, h, &kv_full[st]);
          tma_load_3d(vd + hf * kHalf, &tmV, 64 * hf, y, h, &kv_full[st]);
        }
      }
    }
  } else if (warp == kSoftmaxWarps + 1) {
    // ---------------------------------------------------------- MMA issuer
    // order: S0, S1, then per block i: P.V of i, S of i+2 (into the buffer
    // P.V of i reads; the MMA pipe keeps the two in order)
    if (lane == 0 && nb > 0) {
      constexpr uint32_t idQK = idesc_f16kind(!F16QK, false, kBN);
      constexpr uint32_t idPV = idesc_f16kind(!F16P, true, D);
      const uint32_t q_s = smem_u32(smem + SM::kOffQ);
      bool ok = mbar_wait(q_full, 0, &misc[1]);
      auto issue_s = [&](int j) {
        const int st = j % kStages, b = j & 1;
        if (!mbar_wait(&kv_full[st], (j / kStages) & 1, &misc[1])) return false;
        // no wait for the P.V that last read this buffer: tcgen05.mma from one
        // thread execute in issue order, so these writes follow its reads
        tc_fence_after();
        const uint32_t k_s = smem_u32(smem + SM::kOffK + st * kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_ss(tS(b), sdesc(q_s + off, kHalf, 1024), sdesc(k_s + off, kHalf, 1024), idQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[b]);
        return true;
      };
      auto issue_pv = [&](int i) {
        const int b = i & 1, st = i % kStages;
        if (!mbar_wait(&p_full[b], (i >> 1) & 1, &misc[1])) return false;
        tc_fence_after();
        const uint32_t v_s = smem_u32(smem + SM::kOffV + st * kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // P: 16 keys = 8 packed bf16x2 columns, high part at 16kk, low part at
          // 16kk + 8; V: 16 key rows = two 8-row swizzle atoms
          const uint64_t vd = sdesc(v_s + kk * 2048, kHalf, 1024);
          mma_ts(tO(b), tS(b) + kk * 16, vd, idPV, (i >= 2 || kk > 0) ? 1u : 0u);
          if (!F16P) mma_ts(tO(b), tS(b) + kk * 16 + 8, vd, idPV, 1u);
        }
        mma_commit(&o_done[b]);
        mma_commit(&kv_empty[st]);
        mma_commit(&s_free[b]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nb > 1) ok = issue_s(1);
      for (int i = 0; i < nb && ok; ++i) {
        ok = issue_pv(i);
        if (ok && i + 2 < nb) ok = issue_s(i + 2);
      }
      if (!ok) misc[1] = 1;
    }
  } else {
    // ---------------------------------------------------------- softmax rows
    const int grp = warp / kGroupWarps;                // this group takes blocks grp, grp+2, ...
    const int wq = warp % kGroupWarps;                 // TMEM lane quarter
    const int row = wq * 32 + lane;                    // TMEM lane = tile row
    const long long lin = lin0 + row;
    const bool valid_row = lin < p.rows_h;
    const long long qi = lin % p.n_q;                  // query index within the chunk
    // last visible key index (-1: none), never past the window's last key
    const long long vis_last = valid_row ? min(p.q_pos0 + qi - p.win_pos0, p.win_len - 1) : -1;
    float sc_row = p.scale_log2;                       // log2-domain score scale of this row
    if constexpr (F16QK) {
      if (valid_row) sc_row *= ldexpf(p.qfac[row0 + row], f16_exponent(*p.kmax_bits));
    }
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t sS = tS(grp) + lane_off, sO = tO(grp) + lane_off;
    // l is kept as two partial sums (even and odd keys) for the packed adds
    float m = -INFINITY, la = 0.f, lb = 0.f;
    bool alive = true;
    int k = 0;
    for (int i = grp; i < nb && alive; i += 2, ++k) {
      const int j = jb + i;
      // keep the warp together: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[grp], k & 1, &misc[1]))) { alive = false; misc[1] = 1; break; }
      tc_fence_after();
      const long long k0 = (long long)j * kBN;
      // tcgen05.ld / st are warp-collective: every branch around them below is
      // uniform across the warp (per-row conditions only select values)
      const bool edge = __any_sync(0xffffffffu, k0 + kBN - 1 > vis_last);   // some row crosses the edge
      // pass 1: block maximum (masking only on a block that crosses the edge)
      float mj = -INFINITY;
      if (!edge) {
        // four independent running maxima: a single chain of 64 dependent
        // max instructions would set the pace of this pass
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(sS + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            mx0 = max3(mx0, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
            mx1 = max3(mx1, __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
            mx2 = max3(mx2, __uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
            mx3 = max3(mx3, __uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
          }
        }
        mj = max3(mx0, mx1, fmaxf(mx2, mx3));
      } else {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(sS + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (k0 + c * 32 + e <= vis_last) mj = fmaxf(mj, __uint_as_float(v[e]));
        }
      }
      mj *= sc_row;
      const bool move = mj > m + kRescaleThreshold || (m == -INFINITY && mj != -INFINITY);
      const bool scale_o = move && m != -INFINITY;
      if (__any_sync(0xffffffffu, scale_o)) {
        // the scores of this block being complete implies this group's
        // previous P.V is complete too (all earlier MMAs were committed)
        const float r = scale_o ? fast_exp2(m - mj) : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(sO + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * r);
          tmem_st32(sO + c * 32, v);
        }
        tmem_wait_st();
        la *= r;
        lb *= r;
      }
      if (move) m = mj;
      // pass 2: P over the consumed scores -- fp16 P * 2^7 (at most 2^15 under
      // the 2^8 rescale threshold; l is summed in the same units), or a bf16
      // pair hi + lo (P.V then carries about 16 significant bits of P).  A
      // fully masked block has m = -inf and yields P = 0 through the mask below.
      const float sc = sc_row;
      const float mm = (m == -INFINITY) ? 0.f : m - kPBias;
      const long long lim = edge ? vis_last - k0 : (long long)kBN;   // keys e <= lim are visible
#pragma unroll 2
      for (int c = 0; c < kBN / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(sS + c * 16, v);
        tmem_wait_ld();
        uint32_t vh[8], vl[8];
        if (!edge && m != -INFINITY) {   // per-row branch: math only
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // a key pair's exponents and sums in packed f32x2 instructions
            float x0, x1;
            f2_fma(x0, x1, __uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]), sc, sc, -mm, -mm);
            const float p0 = fast_exp2(x0);
            const float p1 = fast_exp2(x1);
            if (F16P) {
              vh[e] = pack_f16x2(p0, p1);
            } else {
              const uint32_t hi = pack_bf16x2(p0, p1);
              vh[e] = hi;
              vl[e] = pack_bf16x2(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xFFFF0000u));
            }
            f2_add(la, lb, la, lb, p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const bool ok0 = (m != -INFINITY) && (c * 16 + 2 * e <= lim);
            const bool ok1 = (m != -INFINITY) && (c * 16 + 2 * e + 1 <= lim);
            const float p0 = ok0 ? fast_exp2(fmaf(__uint_as_float(v[2 * e]), sc, -mm)) : 0.f;
            const float p1 = ok1 ? fast_exp2(fmaf(__uint_as_float(v[2 * e + 1]), sc, -mm)) : 0.f;
            if (F16P) {
              vh[e] = pack_f16x2(p0, p1);
            } else {
              const uint32_t hi = pack_bf16x2(p0, p1);
              vh[e] = hi;
              vl[e] = pack_bf16x2(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xFFFF0000u));
            }
            f2_add(la, lb, la, lb, p0, p1);
          }
        }
        // keys 16c .. 16c+15: (high part) in columns 16c .. 16c+7, low part in
        // 16c+8 .. 16c+15 -- exactly the columns just read, never unread ones
        tmem_st8(sS + c * 16, vh);
        if (!F16P) tmem_st8(sS + c * 16 + 8, vl);
      }
      // every lane's P stores have completed (wait::st) before the warp's one
      // arrival releases them to the MMA thread
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[grp]);
    }
    const float l = la + lb;
    // ---- this group's last P.V
    const int nk = (nb > grp) ? (nb - grp + 1) / 2 : 0;   // blocks this group owned
    if (alive && nk > 0) {
      if (!mbar_wait(&o_done[grp], (nk - 1) & 1, &misc[1])) misc[1] = 1;
      tc_fence_after();
    }
    if (grp == 1) ml1[row] = make_float2(nk > 0 ? m - kPBias : -INFINITY, nk > 0 ? l : 0.f);
    tc_fence_before();
    group_bar(1);
    if (grp == 0) {
      // ---- epilogue: combine both groups, fold this window into the accumulator
      tc_fence_after();
      const float2 o1ml = ml1[row];
      const int nk1 = (nb > 1) ? nb / 2 : 0;
      // references in the units l was summed in (P scaled by 2^kPBias)
      const float m0v = nk > 0 ? m - kPBias : -INFINITY, l0v = nk > 0 ? l : 0.f;
      const float M = fmaxf(m0v, o1ml.x);
      const float vsc = F16P ? ldexpf(1.f, f16_exponent(*p.vmax_bits)) : 1.f;   // undo V's 2^-e
      const float w0 = (m0v == -INFINITY) ? 0.f : fast_exp2(m0v - M);
      const float w1 = (o1ml.x == -INFINITY) ? 0.f : fast_exp2(o1ml.x - M);
      const float lt = l0v * w0 + o1ml.y * w1;
      const bool have = alive && lt > 0.f;
      const long long orow = row0 + row;               // = (query head) * n_q + qi
      const uint32_t o0a = tO(0) + lane_off, o1a = tO(1) + lane_off;
      if (p.nsplit > 1) {
        // partial of this key range: normalised o and its lse2, folded later
        const size_t part = ((size_t)h * p.n_tiles + tile) * p.nsplit + split;
        float* po = p.ws_o + (part * kBM + row) * D;
        const float inv = have ? vsc / lt : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t v0[16], v1[16];
          if (nk > 0) tmem_ld16(o0a + c * 16, v0);     // nk, nk1 are uniform across the CTA
          if (nk1 > 0) tmem_ld16(o1a + c * 16, v1);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            float ov[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float x = 0.f;
              if (have) {
                if (nk > 0) x += w0 * __uint_as_float(v0[e + u]);
                if (nk1 > 0) x += w1 * __uint_as_float(v1[e + u]);
              }
              ov[u] = x * inv;
            }
            *reinterpret_cast<float4*>(po + c * 16 + e) = make_float4(ov[0], ov[1], ov[2], ov[3]);
          }
        }
        p.ws_lse[part * kBM + row] = have ? M + log2f(lt) : -INFINITY;
      } else {
        // every lane runs the (warp-collective) TMEM loads; rows past the
        // head's last row neither read nor write the accumulator
        float* ao = p.acc_o + orow * D;
        const float lse = have ? M + log2f(lt) : -INFINITY;
        const float La = (p.fold && valid_row) ? p.acc_lse2[orow] : -INFINITY;
        float wa = 0.f, wb = 0.f, L = -INFINITY;
        if (have) {
          if (La == -INFINITY) {
            wb = vsc / lt;
            L = lse;
          } else {
            const float Mx = fmaxf(La, lse);
            L = Mx + log2f(exp2f(La - Mx) + exp2f(lse - Mx));
            wa = exp2f(La - L);
            wb = exp2f(lse - L) * vsc / lt;
          }
        } else {
          wa = 1.f;
          L = La;
        }
        const bool write = valid_row && (have || !p.fold);
  #pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t v0[16], v1[16];
          if (nk > 0) tmem_ld16(o0a + c * 16, v0);     // nk, nk1 are uniform across the CTA
          if (nk1 > 0) tmem_ld16(o1a + c * 16, v1);
          tmem_wait_ld();
  #pragma unroll
          for (int e = 0; e < 16; e += 4) {
            float ov[4];
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              float x = 0.f;
              if (have) {
                if (nk > 0) x += w0 * __uint_as_float(v0[e + u]);
                if (nk1 > 0) x += w1 * __uint_as_float(v1[e + u]);
              }
              ov[u] = x * wb;
            }
            if (write) {
              float4 a = (p.fold && wa != 0.f) ? *reinterpret_cast<const float4*>(ao + c * 16 + e)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
              float4 o = make_float4(wa * a.x + ov[0], wa * a.y + ov[1], wa * a.z + ov[2], wa * a.w + ov[3]);
              *reinterpret_cast<float4*>(ao + c * 16 + e) = o;
            }
          }
        }
        if (write) p.acc_lse2[orow] = L;
      }
    }
  }

  // ---- teardown: every tcgen05 op of the CTA has completed (both groups
  // waited for their last P.V); the allocating warp frees TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == kSoftmaxWarps + 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Fold the key-range partials of every row into the accumulator: one warp per
// row, each of the first D / 4 lanes a float4 of the D dims.  Same arithmetic
// as the direct epilogue: L = max + log2(sum of 2^(lse - max)),
// o = sum of 2^(lse - L) o_s.
constexpr int kFoldWarps = 8;
template <int D>
__global__ void __launch_bounds__(32 * kFoldWarps) prefill_fold_kernel(const PParams p, long long n_rows) {
  const long long r = (long long)blockIdx.x * kFoldWarps + (threadIdx.x >> 5);   // = h * rows_h + lin
  const int lane = threadIdx.x & 31;
  if (r >= n_rows || lane >= D / 4) return;
  const long long hh = r / p.rows_h, lin = r - hh * p.rows_h;
  const long long tile_lin = hh * p.n_tiles + lin / kBM;
  const int row = (int)(lin % kBM);
  const float* pl = p.ws_lse + (size_t)tile_lin * p.nsplit * kBM + row;
  const float La = p.fold ? p.acc_lse2[r] : -INFINITY;
  float M = La;
  for (int s2 = 0; s2 < p.nsplit; ++s2) M = fmaxf(M, pl[(size_t)s2 * kBM]);
  float4* ao = reinterpret_cast<float4*>(p.acc_o + r * D) + lane;
  if (M == -INFINITY) {  // nothing visible anywhere: o = 0, lse2 = -inf (kept when folding)
    if (!p.fold) {
      *ao = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) p.acc_lse2[r] = -INFINITY;
    }
    return;
  }
  float sum = (La == -INFINITY) ? 0.f : exp2f(La - M);
  for (int s2 = 0; s2 < p.nsplit; ++s2) {
    const float ls = pl[(size_t)s2 * kBM];
    if (ls != -INFINITY) sum += exp2f(ls - M);
  }
  const float L = M + log2f(sum);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  if (La != -INFINITY) {
    const float wa = exp2f(La - L);
    const float4 a = *ao;
    o = make_float4(wa * a.x, wa * a.y, wa * a.z, wa * a.w);
  }
  const float4* po = reinterpret_cast<const float4*>(p.ws_o + ((size_t)tile_lin * p.nsplit * kBM + row) * D) + lane;
  for (int s2 = 0; s2 < p.nsplit; ++s2) {
    const float ls = pl[(size_t)s2 * kBM];
    if (ls == -INFINITY) continue;
    const float w = exp2f(ls - L);
    const float4 x = po[(size_t)s2 * kBM * (D / 4)];
    o.x += w * x.x;
    o.y += w * x.y;
    o.z += w * x.z;
    o.w += w * x.w;
  }
  *ao = o;
  if (lane == 0) p.acc_lse2[r] = L;
}

// ---------------------------------------------------------------- fp16 V
// max |v| over the window (bf16 element (h, j, d) at h * stride + j * D + d):
// per-block reduction, one atomicMax on the bit pattern (non-negative floats
// order like their bits).
__global__ void __launch_bounds__(256) v16_max_kernel(const uint16_t* v, long long stride, long long win_len,
                                                      int D, long long n_vec, uint32_t* vmax) {
  __shared__ float sh[8];
  float mx = 0.f;
  const long long per_head = win_len * (D / 8);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += (long long)gridDim.x * blockDim.x) {
    const long long h = i / per_head, r = i - h * per_head;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(v + h * stride) + r);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx = fmaxf(mx, fabsf(__uint_as_float(w[e] << 16)));
      mx = fmaxf(mx, fabsf(__uint_as_float(w[e] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) mx = fmaxf(mx, sh[w]);
    atomicMax(vmax, __float_as_uint(mx));
  }
}

// V16[h][j][d] = fp16_rn(v * 2^-e); scaling by a power of two is exact
// outside fp16's subnormal range.
__global__ void __launch_bounds__(256) v16_convert_kernel(const uint16_t* v, long long stride, long long win_len,
                                                          int D, long long n_vec, const uint32_t* vmax, uint16_t* v16) {
  const float sc = ldexpf(1.f, -f16_exponent(*vmax));
  const long long per_head = win_len * (D / 8);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += (long long)gridDim.x * blockDim.x) {
    const long long h = i / per_head, r = i - h * per_head;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(v + h * stride) + r);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_f16x2(__uint_as_float(w[e] << 16) * sc, __uint_as_float(w[e] & 0xFFFF0000u) * sc);
    reinterpret_cast<uint4*>(v16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------- host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

static bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t box[3] = {64, (cuuint32_t)kBM, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Key ranges per tile: enough CTAs that whole waves cover every SM, weighed
// against the fixed cost of a CTA (Q load, pipeline fill, epilogue), counted
// here as four key blocks.
static int plan_splits(long long n_tiles_total, long long nb_tile) {
  const long long sms = device_sm_count();
  int best = 1;
  double best_cost = 1e300;
  for (int k = 1; k <= 32; ++k) {
    if (k > 1 && nb_tile / k < 8) break;
    const long long ctas = n_tiles_total * k;
    const long long waves = (ctas + sms - 1) / sms;
    const double cost = (double)waves * ((double)((nb_tile + k - 1) / k) + 4.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = k;
    }
  }
  return best;
}

static argus_status check_geom(const argus_geom* g, int32_t n_q, int64_t win_len) {
  if (!g) return fail(ARGUS_E_INVALID, "prefill: geometry is NULL");
  if (g->n_q_heads <= 0 || g->n_kv_heads <= 0 || g->n_q_heads % g->n_kv_heads)
    return fail(ARGUS_E_INVALID, "prefill: bad head counts");
  if (g->head_dim != 64 && g->head_dim != 128)
    return fail(ARGUS_E_UNSUPPORTED, "prefill: head_dim %d (supported: 64, 128)", g->head_dim);
  if (n_q < 0 || win_len < 0) return fail(ARGUS_E_INVALID, "prefill: negative n_q or win_len");
  if ((long long)g->n_q_heads * n_q > (1LL << 31) - kBM || win_len > (1LL << 31) - kBN)
    return fail(ARGUS_E_UNSUPPORTED, "prefill: sizes beyond 2^31 rows");
  return ARGUS_OK;
}

// query tiles of one KV head (its G heads' rows stacked)
static long long tiles_per_head(const argus_geom* g, int32_t n_q) {
  return ((long long)(g->n_q_heads / g->n_kv_heads) * n_q + kBM - 1) / kBM;
}

static size_t up16(size_t x) { return (x + 15) / 16 * 16; }

static size_t split_bytes(long long n_tiles_total, int nsplit, int D) {
  return nsplit > 1 ? (size_t)n_tiles_total * nsplit * kBM * (D + 1) * sizeof(float) : 0;
}

// fp16 copy of one operand over the window: [Hkv][win_len][D]
static size_t win16_bytes(long long n_kv_heads, long long win_len, int D) {
  return (size_t)n_kv_heads * std::max<long long>(win_len, 1) * D * 2;
}

// With a workspace, P.V runs in fp16: after the partials come the window's V
// as scaled fp16 [Hkv][win_len][D] and the max-|v| word.
static size_t ws_total(long long n_tiles_total, int nsplit, long long n_kv_heads, long long win_len, int D) {
  return split_bytes(n_tiles_total, nsplit, D) + win16_bytes(n_kv_heads, win_len, D) + 16;
}

// Staged paged window: partials, fp16 K, fp16 V, fp16 Q [Hq * n_q][D], the
// per-row query factors, then the max-|k| and max-|v| words.
struct PagedWs {
  size_t part, k16, v16, q16, qfac, words, total;
};
static PagedWs paged_ws(const argus_geom* g, int32_t n_q, long long win_len, long long n_tiles_total, int nsplit) {
  PagedWs w;
  const long long rows = (long long)g->n_q_heads * n_q;
  const int D = g->head_dim;
  w.part = 0;
  w.k16 = split_bytes(n_tiles_total, nsplit, D);
  w.v16 = w.k16 + win16_bytes(g->n_kv_heads, win_len, D);
  w.q16 = w.v16 + win16_bytes(g->n_kv_heads, win_len, D);
  w.qfac = w.q16 + up16((size_t)std::max<long long>(rows, 1) * D * 2);
  w.words = w.qfac + up16((size_t)std::max<long long>(rows, 1) * 4);
  w.total = w.words + 16;
  return w;
}

static int resolve_splits(long long tiles, long long win_len, int32_t num_splits, bool have_ws) {
  if (num_splits > 0) return num_splits;
  return have_ws ? plan_splits(tiles, (win_len + kBN - 1) / kBN) : 1;
}

// Tensor maps over Q [rows][D] and K, V [Hkv][rows of a window][D] (element
// strides in elements), all in `dtype`; a window of 0 keys maps one row.  The
// box is 64 dims x 128 rows: one swizzled half of a tile.
static argus_status make_maps(CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv, int D, const void* q,
                              long long q_rows, const void* k, const void* v, long long n_kv_heads,
                              long long win_len, long long kv_stride, CUtensorMapDataType qdt,
                              CUtensorMapDataType kdt, CUtensorMapDataType vdt, long long v_stride) {
  const long long wl = std::max<long long>(win_len, 1);
  const cuuint64_t qd[2] = {(cuuint64_t)D, (cuuint64_t)std::max<long long>(q_rows, 1)};
  const cuuint64_t qs[1] = {(cuuint64_t)D * 2};
  const cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)wl, (cuuint64_t)n_kv_heads};
  const cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)kv_stride * 2};
  const cuuint64_t vs[2] = {(cuuint64_t)D * 2, (cuuint64_t)v_stride * 2};
  if (!make_map(mq, q, 2, qd, qs, qdt)) return fail(ARGUS_E_LAUNCH, "prefill: tensor map for q failed");
  if (!make_map(mk, k, 3, kd, ks, kdt)) return fail(ARGUS_E_LAUNCH, "prefill: tensor map for k failed");
  if (!make_map(mv, v, 3, kd, vs, vdt)) return fail(ARGUS_E_LAUNCH, "prefill: tensor map for v failed");
  return ARGUS_OK;
}

template <int D>
static cudaError_t set_smem_attributes() {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<0, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_kernel<1, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D>::kBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_kernel<2, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<D>::kBytes);
  return e;
}

template <int D>
static void launch_mode(int mode, dim3 grid, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const PParams& p, cudaStream_t s) {
  constexpr int smem = Smem<D>::kBytes;
  if (mode == 0) prefill_kernel<0, D><<<grid, kThreads, smem, s>>>(mq, mk, mv, p);
  else if (mode == 1) prefill_kernel<1, D><<<grid, kThreads, smem, s>>>(mq, mk, mv, p);
  else prefill_kernel<2, D><<<grid, kThreads, smem, s>>>(mq, mk, mv, p);
}

// Launch the attention kernel of `mode` over (tiles, Hkv, splits) and, with
// more than one split, the fold of the partials.
static argus_status launch_attention(int mode, int D, const CUtensorMap& mq, const CUtensorMap& mk,
                                     const CUtensorMap& mv, const PParams& p, long long n_kv_heads, long long n_rows,
                                     cudaStream_t s) {
  static PerContext configured;
  argus_status sta = configured.ensure([](int) {
    cudaError_t e = set_smem_attributes<128>();
    if (e == cudaSuccess) e = set_smem_attributes<64>();
    if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "prefill: smem attribute: %s", cudaGetErrorString(e));
    return ARGUS_OK;
  });
  if (sta != ARGUS_OK) return sta;
  dim3 grid(p.n_tiles, (unsigned)n_kv_heads, p.nsplit);
  if (D == 64) launch_mode<64>(mode, grid, mq, mk, mv, p, s);
  else launch_mode<128>(mode, grid, mq, mk, mv, p, s);
  argus_status st = launch_status("window prefill attention");
  if (st != ARGUS_OK || p.nsplit == 1) return st;
  const unsigned blocks = (unsigned)((n_rows + kFoldWarps - 1) / kFoldWarps);
  if (D == 64) prefill_fold_kernel<64><<<blocks, 32 * kFoldWarps, 0, s>>>(p, n_rows);
  else prefill_fold_kernel<128><<<blocks, 32 * kFoldWarps, 0, s>>>(p, n_rows);
  return launch_status("window prefill attention (fold)");
}

static argus_status common_args(const argus_geom* g, int32_t n_q, int64_t win_len, float softmax_scale, int32_t fold,
                                int32_t num_splits) {
  argus_status st0 = check_geom(g, n_q, win_len);
  if (st0 != ARGUS_OK) return st0;
  if (fold != 0 && fold != 1) return fail(ARGUS_E_INVALID, "prefill: fold must be 0 or 1");
  // the lazy running maximum takes the largest raw score as the largest scaled one
  if (!std::isfinite(softmax_scale) || softmax_scale < 0.f)
    return fail(ARGUS_E_INVALID, "prefill: softmax_scale must be finite and >= 0");
  if (num_splits < 0 || num_splits > 1024) return fail(ARGUS_E_INVALID, "prefill: num_splits out of range");
  return ARGUS_OK;
}

static PParams base_params(const argus_geom* g, int32_t n_q, int64_t win_len, int64_t win_pos0, int64_t q_pos0,
                           float softmax_scale, float* acc_o, float* acc_lse2, int32_t fold) {
  PParams p{};
  p.G = g->n_q_heads / g->n_kv_heads;
  p.n_q = n_q;
  p.rows_h = (long long)p.G * n_q;
  p.n_tiles = (int)tiles_per_head(g, n_q);
  p.win_len = win_len;
  p.win_pos0 = win_pos0;
  p.q_pos0 = q_pos0;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.acc_o = acc_o;
  p.acc_lse2 = acc_lse2;
  p.fold = fold;
  return p;
}

// ---------------------------------------------------------------- staging
// A window of a paged, mixed-codec cache staged into fp16 copies: element
// (h, j, d) of K (or V) is position win_pos0 + j of the sequence, found in
// logical page pos / P, row pos % P, whose codec and slot come from
// page_codec / block_table.  Values are dequantised exactly as the pool defines
// them (codes x scale; INT4 / INT2 code x s + z in fp32), then scaled by the
// window's power of two and rounded to fp16.
struct SParams {
  int Hkv, P, max_pages, D;
  const uint8_t* codes[ARGUS_INT1_G32 + 1];
  const uint8_t* meta[ARGUS_INT1_G32 + 1];
  long long n_slots[ARGUS_INT1_G32 + 1];
  const uint8_t* page_codec;
  const int32_t* block_table;
  long long win_pos0, win_len, n_vec;   // n_vec = Hkv * win_len * D / 8
  uint16_t* k16;
  uint16_t* v16;
  uint32_t* kmax;
  uint32_t* vmax;
  uint32_t* status;
  // query staging
  const uint16_t* q;
  uint16_t* q16;
  float* qfac;
  long long q_rows;
};

__device__ __forceinline__ float f16_to_f32(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xFFFFu)));
}

// Dequantise elements d0 .. d0 + 7 of the key (kv = 0) or value (kv = 1) row at
// sequence position pos for KV head h.  A page whose codec has no pool or whose
// slot lies outside it gives zeros and false.
__device__ __forceinline__ bool stage_load8(const SParams& p, int kv, int h, long long pos, int d0, float (&x)[8]) {
  const long long page = pos / p.P;
  const int row = (int)(pos - page * p.P);
  const int codec = p.page_codec[page];
  const long long slot = p.block_table[page];
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = 0.f;
  if (codec < 0 || codec > ARGUS_INT1_G32 || p.codes[codec] == nullptr || slot < 0 || slot >= p.n_slots[codec])
    return false;
  const size_t unit = ((size_t)slot * 2 + kv) * p.Hkv + h;   // (slot, K|V, head)
  const size_t r = unit * p.P + row;                          // token row of the pool
  const uint8_t* c = p.codes[codec];
  if (codec == ARGUS_FP16 || codec == ARGUS_BF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(c + (r * p.D + d0) * 2);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (codec == ARGUS_BF16) {
        x[2 * e] = __uint_as_float(ww[e] << 16);
        x[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
      } else {
        x[2 * e] = f16_to_f32(ww[e]);
        x[2 * e + 1] = f16_to_f32(ww[e] >> 16);
      }
    }
  } else if (codec == ARGUS_FP8_E4M3 || codec == ARGUS_INT8) {
    const uint2 w = *reinterpret_cast<const uint2*>(c + r * p.D + d0);
    const float sc = reinterpret_cast<const float*>(p.meta[codec])[unit];
    const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (codec == ARGUS_FP8_E4M3) {
        const uint32_t lo = e4m3x2_to_f16x2(ww[e]), hi = e4m3x2_to_f16x2(ww[e] >> 16);
        x[4 * e] = f16_to_f32(lo) * sc;
        x[4 * e + 1] = f16_to_f32(lo >> 16) * sc;
        x[4 * e + 2] = f16_to_f32(hi) * sc;
        x[4 * e + 3] = f16_to_f32(hi >> 16) * sc;
      } else {
#pragma unroll
        for (int b = 0; b < 4; ++b) x[4 * e + b] = (float)(int8_t)((ww[e] >> (8 * b)) & 0xFFu) * sc;
      }
    }
  } else {
    const __half2 sz = reinterpret_cast<const __half2*>(p.meta[codec])[r * (p.D / 32) + d0 / 32];
    const float s = __low2float(sz), z = __high2float(sz);
    if (codec == ARGUS_INT4_G32) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(c + r * (p.D / 2) + d0 / 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fmaf((float)((w >> (4 * e)) & 0xFu), s, z);
    } else if (codec == ARGUS_INT1_G32) {
      const uint32_t w = c[r * (p.D / 8) + d0 / 8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fmaf((float)((w >> e) & 0x1u), s, z);
    } else {
      const uint32_t w = *reinterpret_cast<const uint16_t*>(c + r * (p.D / 4) + d0 / 4);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = fmaf((float)((w >> (2 * e)) & 0x3u), s, z);
    }
  }
  return true;
}

// Vector i of the window: KV head h, window row j, dims d0 .. d0 + 7.
__device__ __forceinline__ void stage_vec(const SParams& p, long long i, int& h, long long& j, int& d0) {
  const int dv = p.D / 8;
  const long long per_head = p.win_len * dv;
  h = (int)(i / per_head);
  const long long rr = i - h * per_head;
  j = rr / dv;
  d0 = (int)(rr - j * dv) * 8;
}

// Pass 1: max |k| and max |v| over the window (block reduction, one atomicMax
// per block on the bit pattern: non-negative floats order like their bits);
// unusable pages are counted once, at their first key vector in the window.
__global__ void __launch_bounds__(256) stage_max_kernel(const SParams p) {
  __shared__ float sh[2][8];
  float mk = 0.f, mv = 0.f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.n_vec; i += (long long)gridDim.x * blockDim.x) {
    int h, d0;
    long long j;
    stage_vec(p, i, h, j, d0);
    const long long pos = p.win_pos0 + j;
    float x[8];
    const bool ok = stage_load8(p, 0, h, pos, d0, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) mk = fmaxf(mk, fabsf(x[e]));
    stage_load8(p, 1, h, pos, d0, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) mv = fmaxf(mv, fabsf(x[e]));
    if (!ok && p.status && h == 0 && d0 == 0 && (j == 0 || pos % p.P == 0)) atomicAdd(p.status, 1u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
  }
  if ((threadIdx.x & 31) == 0) {
    sh[0][threadIdx.x >> 5] = mk;
    sh[1][threadIdx.x >> 5] = mv;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) {
      mk = fmaxf(mk, sh[0][w]);
      mv = fmaxf(mv, sh[1][w]);
    }
    atomicMax(p.kmax, __float_as_uint(mk));
    atomicMax(p.vmax, __float_as_uint(mv));
  }
}

// Pass 2: the scaled fp16 copies of K and V.
__global__ void __launch_bounds__(256) stage_write_kernel(const SParams p) {
  const float sk = ldexpf(1.f, -f16_exponent(*p.kmax));
  const float sv = ldexpf(1.f, -f16_exponent(*p.vmax));
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.n_vec; i += (long long)gridDim.x * blockDim.x) {
    int h, d0;
    long long j;
    stage_vec(p, i, h, j, d0);
    const long long pos = p.win_pos0 + j;
    float x[8];
    uint32_t o[4];
    stage_load8(p, 0, h, pos, d0, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(x[2 * e] * sk, x[2 * e + 1] * sk);
    reinterpret_cast<uint4*>(p.k16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    stage_load8(p, 1, h, pos, d0, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = pack_f16x2(x[2 * e] * sv, x[2 * e + 1] * sv);
    reinterpret_cast<uint4*>(p.v16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The query in fp16: one warp per row of [Hq * n_q][D] bf16, scaled by 2^-e
// from the row's max |q| (into [2^14, 2^15)); qfac[row] = 2^e.
__global__ void __launch_bounds__(256) stage_q_kernel(const SParams p) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.q_rows) return;
  const int lane = threadIdx.x & 31;
  const bool mine = lane < p.D / 4;   // dims 4 lane .. 4 lane + 3
  const uint2 w = mine ? reinterpret_cast<const uint2*>(p.q + row * p.D)[lane] : make_uint2(0u, 0u);
  const float x[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                      __uint_as_float(w.y & 0xFFFF0000u)};
  float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int e = f16_exponent(__float_as_uint(m));
  const float sc = ldexpf(1.f, -e);
  if (mine)
    reinterpret_cast<uint2*>(p.q16 + row * p.D)[lane] =
        make_uint2(pack_f16x2(x[0] * sc, x[1] * sc), pack_f16x2(x[2] * sc, x[3] * sc));
  if (lane == 0) p.qfac[row] = ldexpf(1.f, e);
}

}  // namespace prefill
}  // namespace argus

extern "C" argus_status argus_window_prefill_workspace_bytes(const argus_geom* g, int32_t n_q, int64_t win_len,
                                                             int32_t num_splits, size_t* bytes) {
  using namespace argus::prefill;
  if (!bytes) return argus::fail(ARGUS_E_INVALID, "prefill: bytes is NULL");
  argus_status st = check_geom(g, n_q, win_len);
  if (st != ARGUS_OK) return st;
  if (num_splits < 0 || num_splits > 1024) return argus::fail(ARGUS_E_INVALID, "prefill: num_splits out of range");
  const long long tiles = tiles_per_head(g, n_q) * g->n_kv_heads;
  *bytes = ws_total(tiles, resolve_splits(tiles, win_len, num_splits, true), g->n_kv_heads, win_len, g->head_dim);
  return ARGUS_OK;
}

extern "C" argus_status argus_window_prefill_attn(const argus_geom* g, int32_t n_q, const void* q,
                                                  const void* k, const void* v, int64_t kv_head_stride,
                                                  int64_t win_len, int64_t win_pos0, int64_t q_pos0,
                                                  float softmax_scale, float* acc_o, float* acc_lse2,
                                                  int32_t fold, int32_t num_splits, void* ws, size_t ws_bytes,
                                                  void* stream) {
  using namespace argus;
  using namespace argus::prefill;
  argus_status st0 = common_args(g, n_q, win_len, softmax_scale, fold, num_splits);
  if (st0 != ARGUS_OK) return st0;
  if (n_q == 0) return ARGUS_OK;
  if (!q || !acc_o || !acc_lse2 || (win_len > 0 && (!k || !v)))
    return fail(ARGUS_E_INVALID, "prefill: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(acc_o) | reinterpret_cast<uintptr_t>(ws)) & 15)
    return fail(ARGUS_E_INVALID, "prefill: pointers must be 16-byte aligned");
  const int D = g->head_dim;
  const long long stride = kv_head_stride ? kv_head_stride : win_len * D;
  if (stride % 8 != 0 || stride < win_len * D)
    return fail(ARGUS_E_INVALID, "prefill: kv_head_stride must be >= win_len*head_dim and a multiple of 8");
  PParams p = base_params(g, n_q, win_len, win_pos0, q_pos0, softmax_scale, acc_o, acc_lse2, fold);
  const long long tiles_total = (long long)p.n_tiles * g->n_kv_heads;
  p.nsplit = resolve_splits(tiles_total, win_len, num_splits, ws != nullptr);
  if (p.nsplit > 65535) return fail(ARGUS_E_UNSUPPORTED, "prefill: too many splits");
  const bool f16p = ws != nullptr;
  uint16_t* v16 = nullptr;
  uint32_t* vmax = nullptr;
  if (p.nsplit > 1 || f16p) {
    const size_t need = ws_total(tiles_total, p.nsplit, g->n_kv_heads, win_len, D);
    if (!ws || ws_bytes < need) return fail(ARGUS_E_WORKSPACE, "prefill: workspace %zu < %zu", ws_bytes, need);
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    if (p.nsplit > 1) {
      p.ws_o = reinterpret_cast<float*>(w8);
      p.ws_lse = p.ws_o + (size_t)tiles_total * p.nsplit * kBM * D;
    }
    v16 = reinterpret_cast<uint16_t*>(w8 + split_bytes(tiles_total, p.nsplit, D));
    vmax = reinterpret_cast<uint32_t*>(w8 + split_bytes(tiles_total, p.nsplit, D) + win16_bytes(g->n_kv_heads, win_len, D));
    p.vmax_bits = vmax;
  }
  CUtensorMap mq, mk, mv;
  const void* kk = win_len > 0 ? k : q;
  argus_status stm = f16p ? make_maps(&mq, &mk, &mv, D, q, (long long)g->n_q_heads * n_q, kk, v16, g->n_kv_heads,
                                      win_len, stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                      CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                      std::max<long long>(win_len, 1) * D)
                          : make_maps(&mq, &mk, &mv, D, q, (long long)g->n_q_heads * n_q, kk, win_len > 0 ? v : q,
                                      g->n_kv_heads, win_len, stride, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                      CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, stride);
  if (stm != ARGUS_OK) return stm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (f16p) {
    // the window's V in fp16, scaled by 2^-e from its max |v|
    if (cudaMemsetAsync(vmax, 0, sizeof(uint32_t), s) != cudaSuccess)
      return fail(ARGUS_E_LAUNCH, "prefill: clearing the max word failed");
    const long long n_vec = (long long)g->n_kv_heads * win_len * (D / 8);
    const int blocks = (int)std::max<long long>(1, std::min<long long>((n_vec + 255) / 256, 8LL * device_sm_count()));
    if (win_len > 0) {
      v16_max_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(v), stride, win_len, D, n_vec, vmax);
      v16_convert_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint16_t*>(v), stride, win_len, D, n_vec, vmax, v16);
      argus_status stc = launch_status("argus_window_prefill_attn (fp16 v)");
      if (stc != ARGUS_OK) return stc;
    }
  }
  return launch_attention(f16p ? 1 : 0, D, mq, mk, mv, p, g->n_kv_heads, (long long)g->n_q_heads * n_q, s);
}

extern "C" argus_status argus_paged_window_prefill_workspace_bytes(const argus_geom* g, int32_t n_q, int64_t win_len,
                                                                   int32_t num_splits, size_t* bytes) {
  using namespace argus::prefill;
  if (!bytes) return argus::fail(ARGUS_E_INVALID, "paged prefill: bytes is NULL");
  argus_status st = check_geom(g, n_q, win_len);
  if (st != ARGUS_OK) return st;
  if (num_splits < 0 || num_splits > 1024) return argus::fail(ARGUS_E_INVALID, "prefill: num_splits out of range");
  const long long tiles = tiles_per_head(g, n_q) * g->n_kv_heads;
  *bytes = paged_ws(g, n_q, win_len, tiles, resolve_splits(tiles, win_len, num_splits, true)).total;
  return ARGUS_OK;
}

extern "C" argus_status argus_paged_window_prefill_attn(const argus_geom* g, int32_t n_q, const void* q,
                                                        const argus_pool* pools, int32_t n_pools,
                                                        const uint8_t* page_codec, const int32_t* block_table,
                                                        int32_t max_pages, int64_t win_pos0, int64_t win_len,
                                                        int64_t q_pos0, float softmax_scale, float* acc_o,
                                                        float* acc_lse2, int32_t fold, int32_t num_splits, void* ws,
                                                        size_t ws_bytes, uint32_t* status, void* stream) {
  using namespace argus;
  using namespace argus::prefill;
  argus_status st0 = common_args(g, n_q, win_len, softmax_scale, fold, num_splits);
  if (st0 != ARGUS_OK) return st0;
  if (g->page_tokens <= 0) return fail(ARGUS_E_INVALID, "paged prefill: page_tokens must be positive");
  if (max_pages <= 0 || win_pos0 < 0 || win_pos0 + win_len > (long long)max_pages * g->page_tokens)
    return fail(ARGUS_E_INVALID, "paged prefill: window [%lld, %lld) outside the %d pages of the table",
                (long long)win_pos0, (long long)(win_pos0 + win_len), max_pages);
  if (n_pools < 0 || n_pools > ARGUS_INT1_G32 + 1 || (n_pools > 0 && !pools))
    return fail(ARGUS_E_INVALID, "paged prefill: bad pool list");
  if (n_q == 0) return ARGUS_OK;
  if (!q || !acc_o || !acc_lse2 || !ws || (win_len > 0 && (!page_codec || !block_table)))
    return fail(ARGUS_E_INVALID, "paged prefill: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(acc_o) | reinterpret_cast<uintptr_t>(ws)) & 15)
    return fail(ARGUS_E_INVALID, "paged prefill: q, acc_o and ws must be 16-byte aligned");
  SParams sp{};
  bool seen[ARGUS_INT1_G32 + 1] = {};
  for (int i = 0; i < n_pools; ++i) {
    const argus_pool& pool = pools[i];
    if (pool.codec < 0 || pool.codec > ARGUS_INT1_G32 || seen[pool.codec] || pool.n_slots < 0)
      return fail(ARGUS_E_INVALID, "paged prefill: pool %d (codec %d) invalid or repeated", i, pool.codec);
    seen[pool.codec] = true;
    if (pool.n_slots > 0) {
      if (!pool.codes || (reinterpret_cast<uintptr_t>(pool.codes) & 15))
        return fail(ARGUS_E_INVALID, "paged prefill: pool %d codes NULL or not 16-byte aligned", i);
      if (pool.codec >= ARGUS_FP8_E4M3 && (!pool.meta || (reinterpret_cast<uintptr_t>(pool.meta) & 15)))
        return fail(ARGUS_E_INVALID, "paged prefill: pool %d meta NULL or not 16-byte aligned", i);
    }
    // host pools are staged from host memory with the same plain loads
    const void* dc = nullptr;
    const void* dm = nullptr;
    const argus_status stp = pool_device_ptrs(pool, &dc, &dm);
    if (stp != ARGUS_OK) return stp;
    sp.codes[pool.codec] = static_cast<const uint8_t*>(dc);
    sp.meta[pool.codec] = static_cast<const uint8_t*>(dm);
    sp.n_slots[pool.codec] = pool.n_slots;
  }
  PParams p = base_params(g, n_q, win_len, win_pos0, q_pos0, softmax_scale, acc_o, acc_lse2, fold);
  const long long tiles_total = (long long)p.n_tiles * g->n_kv_heads;
  p.nsplit = resolve_splits(tiles_total, win_len, num_splits, true);
  if (p.nsplit > 65535) return fail(ARGUS_E_UNSUPPORTED, "prefill: too many splits");
  const PagedWs L = paged_ws(g, n_q, win_len, tiles_total, p.nsplit);
  if (ws_bytes < L.total) return fail(ARGUS_E_WORKSPACE, "paged prefill: workspace %zu < %zu", ws_bytes, L.total);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if (p.nsplit > 1) {
    p.ws_o = reinterpret_cast<float*>(w8 + L.part);
    p.ws_lse = p.ws_o + (size_t)tiles_total * p.nsplit * kBM * g->head_dim;
  }
  uint32_t* words = reinterpret_cast<uint32_t*>(w8 + L.words);
  sp.Hkv = g->n_kv_heads;
  sp.P = g->page_tokens;
  sp.max_pages = max_pages;
  sp.D = g->head_dim;
  sp.page_codec = page_codec;
  sp.block_table = block_table;
  sp.win_pos0 = win_pos0;
  sp.win_len = win_len;
  sp.n_vec = (long long)g->n_kv_heads * win_len * (sp.D / 8);
  sp.k16 = reinterpret_cast<uint16_t*>(w8 + L.k16);
  sp.v16 = reinterpret_cast<uint16_t*>(w8 + L.v16);
  sp.kmax = words;
  sp.vmax = words + 1;
  sp.status = status;
  sp.q = static_cast<const uint16_t*>(q);
  sp.q16 = reinterpret_cast<uint16_t*>(w8 + L.q16);
  sp.qfac = reinterpret_cast<float*>(w8 + L.qfac);
  sp.q_rows = (long long)g->n_q_heads * n_q;
  p.kmax_bits = sp.kmax;
  p.vmax_bits = sp.vmax;
  p.qfac = sp.qfac;
  CUtensorMap mq, mk, mv;
  const long long wl = std::max<long long>(win_len, 1);
  argus_status stm = make_maps(&mq, &mk, &mv, sp.D, sp.q16, sp.q_rows, sp.k16, sp.v16, g->n_kv_heads, win_len,
                               wl * sp.D, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                               CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wl * sp.D);
  if (stm != ARGUS_OK) return stm;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(words, 0, 16, s) != cudaSuccess) return fail(ARGUS_E_LAUNCH, "paged prefill: clearing the max words failed");
  const int sms = device_sm_count();
  if (win_len > 0) {
    const int blocks = (int)std::max<long long>(1, std::min<long long>((sp.n_vec + 255) / 256, 8LL * sms));
    stage_max_kernel<<<blocks, 256, 0, s>>>(sp);
    stage_write_kernel<<<blocks, 256, 0, s>>>(sp);
  }
  stage_q_kernel<<<(unsigned)((sp.q_rows + 7) / 8), 256, 0, s>>>(sp);
  argus_status stc = launch_status("argus_paged_window_prefill_attn (staging)");
  if (stc != ARGUS_OK) return stc;
  return launch_attention(2, sp.D, mq, mk, mv, p, g->n_kv_heads, sp.q_rows, s);
}
