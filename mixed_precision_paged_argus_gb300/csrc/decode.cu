// argus_paged_decode_attn: single-token decode attention over a paged KV cache
// whose pages each sit in their own codec tier (FP16 / BF16 / FP8 e4m3 / INT8 /
// INT4 group-32).
//
// Method ("ARGUS: Heterogeneous KV-cache memory management", sections "Why
// decode is slow" and "Direct paged attention"): an exact online softmax
// consumes the cache one page tile at a time through a structure-of-arrays
// page table, with grouped-query attention; nothing context-sized is ever
// materialised.  The block table translates logical pages to physical slots
// and the page list may be the indexer's selection ("feat(kvcache): host-RAM KV
// tier for sparse-attention models", sections "Why this works for sparse
// attention" and "Design").  Context splits are folded by log2-sum-exp.
//
// GB300 design
//  * grid (split, KV head, batch row); 4 consumer warps + 1 producer warp.
//  * The producer walks the split's 16-token chunks, translates each through
//    the block table and streams its K and V rows (plus INT4 group metadata)
//    into a ring of shared-memory stages with 1-D cp.async.bulk copies that
//    complete on mbarriers; every chunk is one contiguous run of a page.
//  * Each consumer warp owns one chunk per stage.  Codes are dequantised in
//    registers straight into m16n8k16 tensor-core fragments: tokens on M, the
//    G <= 8 query heads of the KV head on N, head_dim on K.  FP8 and INT8 codes
//    are exact in fp16, so their per-(page, head) scales are applied outside the
//    MMA (K scale on the scores; V scale folded into the accumulator's running
//    rescale), keeping the dot products exact.
//  * Online softmax in the log2 domain; P is transposed in registers
//    (movmatrix) into the B fragment of the P.V MMA, whose A operand is V^T
//    assembled from pairs of token rows with byte permutes.
//  * Warps merge in shared memory; context splits are folded by a second,
//    fully parallel kernel chained with programmatic dependent launch.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace argus {
namespace decode {

constexpr int kChunk = 16;
constexpr int kChunksPerStage = 8;

// Chunks per ring stage: 8, or 16 in the narrow layout -- launches whose pools
// all hold byte or nibble codes (FP8, INT8, INT4) at head_dim 128, where a
// chunk slot needs half the bytes.
template <bool NARROW>
constexpr int chunks_per_stage() { return NARROW ? 16 : kChunksPerStage; }

// Consumer warps per CTA: head_dim 64 runs 4 warps of two chunks per stage
// (two CTAs per SM; a second chunk in flight per warp hides MMA latency);
// head_dim 128 runs 8 warps, of one chunk (16-bit layout: the ring fills
// shared memory) or two chunks (narrow layout) per stage.
// Producer warps: a warp issues its bulk copies one after another (about 60
// cycles each, whatever their size), so the narrow ring -- 16 chunks and up
// to 64 copies per stage -- has two producers taking alternate batches of two
// stages; 12 warps still fit the register file at the consumers' count.
template <int D, bool NARROW = false>
struct Warps {
  static constexpr int kConsumer = (D == 64) ? 4 : 8;
  static constexpr int kNC = chunks_per_stage<NARROW>() / kConsumer;  // chunks per warp and stage
  static constexpr int kProducers = NARROW ? 3 : 1;
  static constexpr int kBatch = NARROW ? 16 : 32;   // chunks a producer translates per round trip
  static constexpr int kThreads = 32 * (kConsumer + kProducers);
};
constexpr int kMaxG = 8;
constexpr int kNumCodecs = ARGUS_INT1_G32 + 1;
constexpr int kMaxSplits = 512;  // bounds the split combine's per-thread loads
constexpr int kFoldThreads = 256;

enum Family { kFamF16 = 0, kFamBF16 = 1, kFamMixed = 2 };

struct Params {
  int B, Hkv, G, P, max_pages;
  const void* q;
  const uint8_t* codes[kNumCodecs];   // indexed by argus_codec
  const uint8_t* meta[kNumCodecs];
  long long n_slots[kNumCodecs];
  uint32_t host_mask;        // bit c: the pool of codec c lives in host memory
  const uint8_t* page_codec;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* sel_pages;
  const int32_t* sel_count;
  int sel_width;
  float scale_log2;
  void* out;
  int out_bf16;
  float* out_f32;
  float* lse2_out;
  uint32_t* status;
  int cps;         // dense pages: chunks per split, a multiple of kChunksPerStage
  int num_splits;  // grid.x (a selection's entries are dealt round-robin over the splits)
  int pdl;         // 0: stream order; 1: early start, inputs read before the wait;
                   // 2: early start, every input read after the wait
  int window;      // > 0: only the newest `window` tokens and the first `sinks` are visible
  int sinks;
  float* part_o;   // [B][Hkv][num_splits][G][D]
  float* part_lse; // [B][Hkv][num_splits][G]
  unsigned long long wait_ns;  // limit of every mbarrier wait
  int stall_stage; // >= 0 only in the stall test: the producer withholds this
                   // stage's descriptor arrival until the consumers give up
};

struct ChunkDesc {
  int32_t codec;  // -1: empty slot in the stage
  uint32_t vmask; // sliding window: bit r set for each visible row r; otherwise
                  // the number of leading visible rows
  float kscale;
  float vscale;
  // a page of a pool in host memory: the chunk's K and V rows (and INT4 / INT2
  // metadata), read in place by the consuming warp; null for device pages,
  // which the producer copies into the stage
  const uint8_t* hk;
  const uint8_t* hv;
  const uint8_t* hmk;
  const uint8_t* hmv;
};

// Dense chunk list of one sequence of seq_len tokens.  Without a window every
// 16-token chunk is listed.  With window > 0 the visible tokens are the first
// `sinks` and the newest `window` ones: the list is the sink chunks [0, cs)
// followed by the window chunks [cw, ceil(seq_len / 16)), cw >= cs, so that
// list entry v is chunk v (v < cs) or chunk v - cs + cw.
struct ChunkList {
  int n, cs, cw;
  __host__ __device__ int chunk(int v) const { return v < cs ? v : v - cs + cw; }
};

__host__ __device__ inline ChunkList dense_chunks(int seq_len, int window, int sinks) {
  const int nc = (seq_len + kChunk - 1) / kChunk;
  ChunkList cl{nc, nc, nc};
  if (window > 0) {
    const int lo = seq_len > window ? seq_len - window : 0;   // first window token
    cl.cs = sinks > 0 ? min((sinks + kChunk - 1) / kChunk, nc) : 0;
    cl.cw = max(cl.cs, lo / kChunk);
    cl.n = cl.cs + (nc - cl.cw);
  }
  return cl;
}

// Visible rows of the chunk starting at token tok0: bit r for token tok0 + r.
__device__ __forceinline__ uint32_t chunk_rows(int tok0, int seq_len, int window, int sinks) {
  const int nv = seq_len - tok0;
  if (nv <= 0) return 0u;
  uint32_t m = nv >= kChunk ? 0xFFFFu : (1u << nv) - 1u;
  if (window > 0) {
    const long long a = (long long)seq_len - window - tok0;   // rows >= a are inside the window
    const uint32_t win = a <= 0 ? 0xFFFFu : (a >= kChunk ? 0u : (0xFFFFu << (int)a) & 0xFFFFu);
    const int sb = sinks - tok0;              // rows < sb are sink tokens
    const uint32_t snk = sb <= 0 ? 0u : (sb >= kChunk ? 0xFFFFu : (1u << sb) - 1u);
    m &= win | snk;
  }
  return m;
}

template <int D, bool NARROW = false>
struct Layout {
  static constexpr int kCPS = chunks_per_stage<NARROW>();
  static constexpr int kNI = D / 32;                   // 32-dim groups per row
  static constexpr int kKV = kChunk * (NARROW ? 1 : 2) * D;   // K (or V) bytes of a chunk slot
  static constexpr int kMeta = kChunk * kNI * 4;       // INT4 {scale, zero} of a chunk
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kKV;
  static constexpr int kOffMK = 2 * kKV;
  static constexpr int kOffMV = 2 * kKV + kMeta;
  static constexpr int kChunkBytes = 2 * kKV + 2 * kMeta;
  static constexpr int kStageBytes = kCPS * kChunkBytes;
  static constexpr int kStages = 3;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kDescOff = kBarOff + 2 * kStages * 8;
  static constexpr int kMiscOff = kDescOff + kStages * kCPS * (int)sizeof(ChunkDesc);
  static constexpr int kSmemBytes = kMiscOff + 64;
  static_assert(kMiscOff % 8 == 0, "misc holds an mbarrier at byte 8");
  static constexpr int kMinBlocks = (D == 128) ? 1 : 2;  // by shared memory
};

// Bytes of one token row of one head in a pool of `codec`.
__host__ __device__ constexpr int row_bytes(int codec, int D) {
  return codec <= ARGUS_BF16 ? 2 * D
       : codec == ARGUS_INT4_G32 ? D / 2
       : codec == ARGUS_INT2_G32 ? D / 4
       : codec == ARGUS_INT1_G32 ? D / 8 : D;
}

// codecs stored as per-group {scale, zero} affine codes
__host__ __device__ constexpr bool affine_codec(int codec) {
  return codec == ARGUS_INT4_G32 || codec == ARGUS_INT2_G32 || codec == ARGUS_INT1_G32;
}

template <int CW>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory");
}

__device__ __forceinline__ int codec_family(int codec) { return codec == ARGUS_BF16 ? 1 : 0; }

__device__ __forceinline__ uint32_t f16_magic_pair(uint32_t u, uint32_t sel) {
  // bytes of u (already biased to unsigned) -> f16 (1024 + byte) pairs
  return prmt(u, 0x64646464u, sel);
}

// K fragments of one chunk: a[c][0..3] are the m16n8k16 A registers of k-chunk
// c for token rows r and r + 8.  Inside each 8-element run of head_dim held by
// a lane, k positions (2t, 2t+1, 2t+8, 2t+9) of k-chunk 2i+hh map to elements
// (2hh, 2hh+4, 2hh+1, 2hh+5); the query fragments use the same map.
// INT4 pages give the raw codes (exact in fp16) and each row's per-group
// {scale, zero} in kz, so that the scores can be formed exactly as
// sum_g scale_g * (q_g . c_g) + zero_g * sum(q_g).
template <int D, bool NARROW>
__device__ __forceinline__ void load_k_frags(int codec, const uint8_t* chunk, int r, int t,
                                             uint32_t (&a)[D / 16][4], float (&kz)[2][D / 32][2]) {
  using L = Layout<D, NARROW>;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = r + 8 * rr;
    if (codec == ARGUS_FP16 || codec == ARGUS_BF16) {
#pragma unroll
      for (int i = 0; i < L::kNI; ++i) {
        const uint4 x = *reinterpret_cast<const uint4*>(chunk + L::kOffK + row * 2 * D + 64 * i + 16 * t);
        a[2 * i][rr] = prmt(x.x, x.z, 0x5410);
        a[2 * i][2 + rr] = prmt(x.x, x.z, 0x7632);
        a[2 * i + 1][rr] = prmt(x.y, x.w, 0x5410);
        a[2 * i + 1][2 + rr] = prmt(x.y, x.w, 0x7632);
      }
    } else if (codec == ARGUS_FP8_E4M3 || codec == ARGUS_INT8) {
      // byte codes: lane t holds dims [64j + 16t, 64j + 16t + 16); word cc of
      // that run feeds k-chunk 4j + cc (bytes 0,1 -> k 2t, 2t+1; bytes 2,3 ->
      // k 2t+8, 2t+9), matching the query fragments qf8.  16-byte loads halve
      // the shared-memory wavefronts of the 8-byte layout.
#pragma unroll
      for (int j = 0; j < D / 64; ++j) {
        const uint4 x = *reinterpret_cast<const uint4*>(chunk + L::kOffK + row * D + 64 * j + 16 * t);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (codec == ARGUS_FP8_E4M3) {
            a[4 * j + cc][rr] = e4m3x2_to_f16x2(w[cc]);
            a[4 * j + cc][2 + rr] = e4m3x2_to_f16x2(w[cc] >> 16);
          } else {
            const uint32_t u = w[cc] ^ 0x80808080u;
            const uint32_t bias = 0x64806480u;  // 1152 = 1024 + 128
            a[4 * j + cc][rr] = hsub2_u32(f16_magic_pair(u, 0x4140), bias);
            a[4 * j + cc][2 + rr] = hsub2_u32(f16_magic_pair(u, 0x4342), bias);
          }
        }
      }
    } else if (codec == ARGUS_INT1_G32) {
      // the lane's 8-element run of group i is one byte, element e at bit e;
      // B | B << 12 puts bit e in the low half and bit e + 4 at bit 16 + e, so
      // shifts of 0..3 give the element pairs (0,4) .. (3,7) of the INT4 map
#pragma unroll
      for (int i = 0; i < L::kNI; ++i) {
        const uint32_t b8 = *(chunk + L::kOffK + row * (D / 8) + 4 * i + t);
        const uint32_t w = b8 | (b8 << 12);
        const __half2 mz = *reinterpret_cast<const __half2*>(chunk + L::kOffMK + (row * L::kNI + i) * 4);
        kz[rr][i][0] = __low2float(mz);
        kz[rr][i][1] = __high2float(mz);
        const uint32_t magic = 0x64006400u;
        a[2 * i][rr] = hsub2_u32(lop3_and_or(w, 0x00010001u, magic), magic);
        a[2 * i][2 + rr] = hsub2_u32(lop3_and_or(w >> 1, 0x00010001u, magic), magic);
        a[2 * i + 1][rr] = hsub2_u32(lop3_and_or(w >> 2, 0x00010001u, magic), magic);
        a[2 * i + 1][2 + rr] = hsub2_u32(lop3_and_or(w >> 3, 0x00010001u, magic), magic);
      }
    } else if (codec == ARGUS_INT2_G32) {
      // the lane's 8-element run of group i is 2 bytes: byte b holds elements
      // 4b .. 4b+3 in bit pairs; spread to the two halves, shifts of 0, 2, 4, 6
      // give the element pairs (0,4), (1,5), (2,6), (3,7) of the INT4 map
#pragma unroll
      for (int i = 0; i < L::kNI; ++i) {
        const uint32_t w16 = *reinterpret_cast<const uint16_t*>(chunk + L::kOffK + row * (D / 4) + 8 * i + 2 * t);
        const uint32_t w = prmt(w16, 0u, 0x4140);
        const __half2 mz = *reinterpret_cast<const __half2*>(chunk + L::kOffMK + (row * L::kNI + i) * 4);
        kz[rr][i][0] = __low2float(mz);
        kz[rr][i][1] = __high2float(mz);
        const uint32_t magic = 0x64006400u;
        a[2 * i][rr] = hsub2_u32(lop3_and_or(w, 0x00030003u, magic), magic);
        a[2 * i][2 + rr] = hsub2_u32(lop3_and_or(w >> 2, 0x00030003u, magic), magic);
        a[2 * i + 1][rr] = hsub2_u32(lop3_and_or(w >> 4, 0x00030003u, magic), magic);
        a[2 * i + 1][2 + rr] = hsub2_u32(lop3_and_or(w >> 6, 0x00030003u, magic), magic);
      }
    } else {  // INT4 group 32
#pragma unroll
      for (int i = 0; i < L::kNI; ++i) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(chunk + L::kOffK + row * (D / 2) + 16 * i + 4 * t);
        const __half2 mz = *reinterpret_cast<const __half2*>(chunk + L::kOffMK + (row * L::kNI + i) * 4);
        kz[rr][i][0] = __low2float(mz);
        kz[rr][i][1] = __high2float(mz);
        const uint32_t magic = 0x64006400u;
        a[2 * i][rr] = hsub2_u32(lop3_and_or(w, 0x000F000Fu, magic), magic);
        a[2 * i][2 + rr] = hsub2_u32(lop3_and_or(w >> 4, 0x000F000Fu, magic), magic);
        a[2 * i + 1][rr] = hsub2_u32(lop3_and_or(w >> 8, 0x000F000Fu, magic), magic);
        a[2 * i + 1][2 + rr] = hsub2_u32(lop3_and_or(w >> 12, 0x000F000Fu, magic), magic);
      }
    }
  }
}

// V^T fragments of one chunk: v[j][0..3] are the A registers of m-block j of
// the P.V MMA (M = head_dim, K = tokens).  Lane (r, t) holds dims
// [DL*r, DL*r + DL) with m-block j covering dims DL*r + 2j (rows r) and
// DL*r + 2j + 1 (rows r + 8), and token rows 2t, 2t+1 (k 0..7) and 2t+8, 2t+9.
template <int D, bool NARROW>
__device__ __forceinline__ void load_v_frags(int codec, const uint8_t* chunk, int r, int t,
                                             uint32_t (&v)[D / 16][4]) {
  using L = Layout<D, NARROW>;
  constexpr int DL = D / 8;
  const int rows[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
  if (codec == ARGUS_FP16 || codec == ARGUS_BF16) {
    uint32_t w[4][DL / 2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* src = chunk + L::kOffV + rows[q] * 2 * D + 2 * DL * r;
      if constexpr (DL == 16) {
        // odd t read the two 16-byte halves in the other order (fewer bank conflicts)
        const int sw = t & 1;
        const uint4 x0 = *reinterpret_cast<const uint4*>(src + 16 * sw);
        const uint4 x1 = *reinterpret_cast<const uint4*>(src + 16 * (sw ^ 1));
        const uint4 lo = sw ? x1 : x0, hi = sw ? x0 : x1;
        w[q][0] = lo.x; w[q][1] = lo.y; w[q][2] = lo.z; w[q][3] = lo.w;
        w[q][4] = hi.x; w[q][5] = hi.y; w[q][6] = hi.z; w[q][7] = hi.w;
      } else {
        const uint4 x = *reinterpret_cast<const uint4*>(src);
        w[q][0] = x.x; w[q][1] = x.y; w[q][2] = x.z; w[q][3] = x.w;
      }
    }
#pragma unroll
    for (int j = 0; j < D / 16; ++j) {
      v[j][0] = prmt(w[0][j], w[1][j], 0x5410);
      v[j][1] = prmt(w[0][j], w[1][j], 0x7632);
      v[j][2] = prmt(w[2][j], w[3][j], 0x5410);
      v[j][3] = prmt(w[2][j], w[3][j], 0x7632);
    }
  } else if (codec == ARGUS_FP8_E4M3 || codec == ARGUS_INT8) {
    uint32_t w[4][DL / 4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* src = chunk + L::kOffV + rows[q] * D + DL * r;
      if constexpr (DL == 16) {
        const uint4 x = *reinterpret_cast<const uint4*>(src);
        w[q][0] = x.x; w[q][1] = x.y; w[q][2] = x.z; w[q][3] = x.w;
      } else {
        const uint2 x = *reinterpret_cast<const uint2*>(src);
        w[q][0] = x.x; w[q][1] = x.y;
      }
    }
#pragma unroll
    for (int k = 0; k < DL / 4; ++k) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int q0 = 2 * half;  // rows (2t, 2t+1) or (2t+8, 2t+9)
        const uint32_t u = prmt(w[q0][k], w[q0 + 1][k], 0x5140);  // a0 b0 a1 b1
        const uint32_t y = prmt(w[q0][k], w[q0 + 1][k], 0x7362);  // a2 b2 a3 b3
        if (codec == ARGUS_FP8_E4M3) {
          v[2 * k][2 * half + 0] = e4m3x2_to_f16x2(u);
          v[2 * k][2 * half + 1] = e4m3x2_to_f16x2(u >> 16);
          v[2 * k + 1][2 * half + 0] = e4m3x2_to_f16x2(y);
          v[2 * k + 1][2 * half + 1] = e4m3x2_to_f16x2(y >> 16);
        } else {
          const uint32_t bias = 0x64806480u;
          const uint32_t ub = u ^ 0x80808080u, yb = y ^ 0x80808080u;
          v[2 * k][2 * half + 0] = hsub2_u32(f16_magic_pair(ub, 0x4140), bias);
          v[2 * k][2 * half + 1] = hsub2_u32(f16_magic_pair(ub, 0x4342), bias);
          v[2 * k + 1][2 * half + 0] = hsub2_u32(f16_magic_pair(yb, 0x4140), bias);
          v[2 * k + 1][2 * half + 1] = hsub2_u32(f16_magic_pair(yb, 0x4342), bias);
        }
      }
    }
  } else if (codec == ARGUS_INT1_G32) {
    // the lane's DL elements of a row are DL/8 bytes (DL = 16: two bytes)
    uint32_t cw[4];
    uint32_t m[4];
    const int grp = (DL * r) / 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* src = chunk + L::kOffV + rows[q] * (D / 8) + (DL / 8) * r;
      if constexpr (DL == 16) cw[q] = *reinterpret_cast<const uint16_t*>(src);
      else cw[q] = *src;
      m[q] = *reinterpret_cast<const uint32_t*>(chunk + L::kOffMV + (rows[q] * L::kNI + grp) * 4);
    }
    const uint32_t magic = 0x64006400u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int q0 = 2 * half;
      const uint32_t s2 = prmt(m[q0], m[q0 + 1], 0x5410);
      const uint32_t z2 = prmt(m[q0], m[q0 + 1], 0x7632);
#pragma unroll
      for (int b = 0; b < DL / 8; ++b) {
        // byte b of row a to byte 0, of row b to byte 2
        const uint32_t x = prmt(cw[q0], cw[q0 + 1], (uint32_t)(b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12)));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t c = hsub2_u32(lop3_and_or(x >> j, 0x00010001u, magic), magic);
          const int d = 8 * b + j;
          v[d / 2][2 * half + (d & 1)] = hfma2_u32(c, s2, z2);
        }
      }
    }
  } else if (codec == ARGUS_INT2_G32) {
    // the lane's DL elements of a row are DL/4 bytes (DL = 16: one word)
    uint32_t cw[4];
    uint32_t m[4];
    const int grp = (DL * r) / 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* src = chunk + L::kOffV + rows[q] * (D / 4) + (DL / 4) * r;
      if constexpr (DL == 16) cw[q] = *reinterpret_cast<const uint32_t*>(src);
      else cw[q] = *reinterpret_cast<const uint16_t*>(src);
      m[q] = *reinterpret_cast<const uint32_t*>(chunk + L::kOffMV + (rows[q] * L::kNI + grp) * 4);
    }
    const uint32_t magic = 0x64006400u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int q0 = 2 * half;
      const uint32_t s2 = prmt(m[q0], m[q0 + 1], 0x5410);
      const uint32_t z2 = prmt(m[q0], m[q0 + 1], 0x7632);
#pragma unroll
      for (int b = 0; b < DL / 4; ++b) {
        // byte b of row a to byte 0, of row b to byte 2 (bytes 1, 3 are masked off)
        const uint32_t x = prmt(cw[q0], cw[q0 + 1], (uint32_t)(b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12)));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t c = hsub2_u32(lop3_and_or(x >> (2 * j), 0x00030003u, magic), magic);
          const int d = 4 * b + j;
          v[d / 2][2 * half + (d & 1)] = hfma2_u32(c, s2, z2);
        }
      }
    }
  } else {  // INT4
    uint32_t w[4][DL / 8];
    uint32_t m[4];
    const int grp = (DL * r) / 32;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint8_t* src = chunk + L::kOffV + rows[q] * (D / 2) + (DL / 2) * r;
      if constexpr (DL == 16) {
        const uint2 x = *reinterpret_cast<const uint2*>(src);
        w[q][0] = x.x; w[q][1] = x.y;
      } else {
        w[q][0] = *reinterpret_cast<const uint32_t*>(src);
      }
      m[q] = *reinterpret_cast<const uint32_t*>(chunk + L::kOffMV + (rows[q] * L::kNI + grp) * 4);
    }
    const uint32_t magic = 0x64006400u;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int q0 = 2 * half;
      const uint32_t s2 = prmt(m[q0], m[q0 + 1], 0x5410);
      const uint32_t z2 = prmt(m[q0], m[q0 + 1], 0x7632);
#pragma unroll
      for (int k = 0; k < DL / 8; ++k) {
        const uint32_t lo = prmt(w[q0][k], w[q0 + 1][k], 0x5410);  // nibbles 0..3 of a | of b
        const uint32_t hi = prmt(w[q0][k], w[q0 + 1][k], 0x7632);  // nibbles 4..7
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint32_t c0 = hsub2_u32(lop3_and_or(lo >> (4 * s), 0x000F000Fu, magic), magic);
          const uint32_t c1 = hsub2_u32(lop3_and_or(hi >> (4 * s), 0x000F000Fu, magic), magic);
          const int d0 = 8 * k + s, d1 = 8 * k + 4 + s;
          v[d0 / 2][2 * half + (d0 & 1)] = hfma2_u32(c0, s2, z2);
          v[d1 / 2][2 * half + (d1 & 1)] = hfma2_u32(c1, s2, z2);
        }
      }
    }
  }
}

// Scores of NCG chunks of one codec: every fragment load and MMA of the
// group is issued before any result is consumed (the m16n8k16 MMA latency is
// long), with two accumulator chains per chunk.  sv is masked and scaled to
// the log2 domain; kscale and the query exponent are applied here.
template <int D, int CODEC, int NCG, bool BF, bool NARROW, bool EXT>
__device__ __forceinline__ void group_scores(const uint8_t* const* cptr, const ChunkDesc* dsc, int r, int t,
                                             const uint32_t (&qf)[D / 16][2], const uint32_t (&qb)[D / 16][2],
                                             const uint32_t (&qf8)[D / 16][2],
                                             const float (&qgs)[D / 32][2], float f0h, float f1h,
                                             float scale_log2, float (*sv)[4], int c0) {
  constexpr int KC = D / 16;
  const uint32_t rbit = 1u << r;   // EXT: this thread's rows r and r + 8 in the chunk's row mask
  uint32_t a[NCG][KC][4];
  float kz[NCG][2][D / 32][2];
#pragma unroll
  for (int c = 0; c < NCG; ++c) load_k_frags<D, NARROW>(CODEC, cptr[c], r, t, a[c], kz[c]);
  if constexpr (affine_codec(CODEC)) {
    float sg[NCG][D / 32][4];
#pragma unroll
    for (int c = 0; c < NCG; ++c)
#pragma unroll
      for (int i = 0; i < D / 32; ++i) sg[c][i][0] = sg[c][i][1] = sg[c][i][2] = sg[c][i][3] = 0.f;
#pragma unroll
    for (int k = 0; k < KC; ++k)
#pragma unroll
      for (int c = 0; c < NCG; ++c) mma_f16(sg[c][k / 2], a[c][k][0], a[c][k][1], a[c][k][2], a[c][k][3], qf[k][0], qf[k][1]);
#pragma unroll
    for (int c = 0; c < NCG; ++c) {
      // sum_g scale_g * acc_g + zero_g * qsum_g, the two heads of a row in
      // packed f32x2 multiply-adds
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        f2_fma(sc[0], sc[1], kz[c][0][i][0], kz[c][0][i][0], sg[c][i][0], sg[c][i][1], sc[0], sc[1]);
        f2_fma(sc[0], sc[1], kz[c][0][i][1], kz[c][0][i][1], qgs[i][0], qgs[i][1], sc[0], sc[1]);
        f2_fma(sc[2], sc[3], kz[c][1][i][0], kz[c][1][i][0], sg[c][i][2], sg[c][i][3], sc[2], sc[3]);
        f2_fma(sc[2], sc[3], kz[c][1][i][1], kz[c][1][i][1], qgs[i][0], qgs[i][1], sc[2], sc[3]);
      }
      const float f0 = scale_log2 * f0h, f1 = scale_log2 * f1h;
      const uint32_t vk = dsc[c].vmask;
      const bool v0 = EXT ? (vk & rbit) != 0u : r < (int)vk;
      const bool v1 = EXT ? (vk & (rbit << 8)) != 0u : r + 8 < (int)vk;
      sv[c0 + c][0] = v0 ? sc[0] * f0 : -INFINITY;
      sv[c0 + c][1] = v0 ? sc[1] * f1 : -INFINITY;
      sv[c0 + c][2] = v1 ? sc[2] * f0 : -INFINITY;
      sv[c0 + c][3] = v1 ? sc[3] * f1 : -INFINITY;
    }
  } else {
    float sc[NCG][2][4];
#pragma unroll
    for (int c = 0; c < NCG; ++c)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) sc[c][h2][0] = sc[c][h2][1] = sc[c][h2][2] = sc[c][h2][3] = 0.f;
#pragma unroll
    for (int k = 0; k < KC; ++k)
#pragma unroll
      for (int c = 0; c < NCG; ++c) {
        if constexpr (BF) mma_bf16(sc[c][k & 1], a[c][k][0], a[c][k][1], a[c][k][2], a[c][k][3], qb[k][0], qb[k][1]);
        else if constexpr (CODEC == ARGUS_FP8_E4M3 || CODEC == ARGUS_INT8)
          mma_f16(sc[c][k & 1], a[c][k][0], a[c][k][1], a[c][k][2], a[c][k][3], qf8[k][0], qf8[k][1]);
        else mma_f16(sc[c][k & 1], a[c][k][0], a[c][k][1], a[c][k][2], a[c][k][3], qf[k][0], qf[k][1]);
      }
#pragma unroll
    for (int c = 0; c < NCG; ++c) {
      const float fk = scale_log2 * dsc[c].kscale;
      const float f0 = fk * f0h, f1 = fk * f1h;
      const uint32_t vk = dsc[c].vmask;
      const bool v0 = EXT ? (vk & rbit) != 0u : r < (int)vk;
      const bool v1 = EXT ? (vk & (rbit << 8)) != 0u : r + 8 < (int)vk;
      sv[c0 + c][0] = v0 ? (sc[c][0][0] + sc[c][1][0]) * f0 : -INFINITY;
      sv[c0 + c][1] = v0 ? (sc[c][0][1] + sc[c][1][1]) * f1 : -INFINITY;
      sv[c0 + c][2] = v1 ? (sc[c][0][2] + sc[c][1][2]) * f0 : -INFINITY;
      sv[c0 + c][3] = v1 ? (sc[c][0][3] + sc[c][1][3]) * f1 : -INFINITY;
    }
  }
}

// O^T += V^T . (w P)^T for NCG chunks of one codec; all V fragments and P
// transposes are formed before the MMAs.  pw[c] = {p0, p1, p2, p3} already
// multiplied by the chunk's V-scale weight; chunks with skip[c] contribute nothing.
template <int D, int CODEC, int NCG, bool BF, bool NARROW>
__device__ __forceinline__ void group_pv(const uint8_t* const* cptr, int r, int t, const float (*pw)[4],
                                         const bool* skip, float (&acc)[D / 16][4]) {
  constexpr int MB = D / 16;
  uint32_t vf[NCG][MB][4];
  uint32_t bh[NCG][2], bl[NCG][2];
#pragma unroll
  for (int c = 0; c < NCG; ++c) {
    load_v_frags<D, NARROW>(CODEC, cptr[c], r, t, vf[c]);
    if constexpr (BF) {
      const float* q = pw[c];
      const uint32_t h01 = pack_bf16x2(q[0], q[1]), h23 = pack_bf16x2(q[2], q[3]);
      const uint32_t l01 = pack_bf16x2(q[0] - __uint_as_float(h01 << 16), q[1] - __uint_as_float(h01 & 0xFFFF0000u));
      const uint32_t l23 = pack_bf16x2(q[2] - __uint_as_float(h23 << 16), q[3] - __uint_as_float(h23 & 0xFFFF0000u));
      bh[c][0] = movmatrix_trans(h01);
      bh[c][1] = movmatrix_trans(h23);
      bl[c][0] = movmatrix_trans(l01);
      bl[c][1] = movmatrix_trans(l23);
    } else {
      bh[c][0] = movmatrix_trans(pack_f16x2(pw[c][0], pw[c][1]));
      bh[c][1] = movmatrix_trans(pack_f16x2(pw[c][2], pw[c][3]));
    }
  }
#pragma unroll
  for (int c = 0; c < NCG; ++c) {
    if (skip[c]) continue;
#pragma unroll
    for (int j = 0; j < MB; ++j) {
      if constexpr (BF) {
        mma_bf16(acc[j], vf[c][j][0], vf[c][j][1], vf[c][j][2], vf[c][j][3], bh[c][0], bh[c][1]);
        mma_bf16(acc[j], vf[c][j][0], vf[c][j][1], vf[c][j][2], vf[c][j][3], bl[c][0], bl[c][1]);
      } else {
        mma_f16(acc[j], vf[c][j][0], vf[c][j][1], vf[c][j][2], vf[c][j][3], bh[c][0], bh[c][1]);
      }
    }
  }
}

// A chunk of a page in host memory, copied into its stage slot by the warp that
// consumes it: K and V rows (16 x row bytes each) as one run of 16-byte vectors
// over the lanes, eight loads per lane in flight before their stores, then the
// INT4 / INT2 group metadata.  Plain loads: the pages are read in place over
// the host link.
template <int D, bool NARROW>
__device__ __forceinline__ void copy_host_chunk(const ChunkDesc& d, uint8_t* slot, int lane) {
  using L = Layout<D, NARROW>;
  const int rowb = row_bytes(d.codec, D);
  const int n16 = kChunk * rowb / 16;          // 16-byte vectors of K (and of V)
  const uint4* srcK = reinterpret_cast<const uint4*>(d.hk);
  const uint4* srcV = reinterpret_cast<const uint4*>(d.hv);
  uint4* dstK = reinterpret_cast<uint4*>(slot + L::kOffK);
  uint4* dstV = reinterpret_cast<uint4*>(slot + L::kOffV);
  for (int base = 0; base < 2 * n16; base += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = base + lane + 32 * i;
      if (idx < 2 * n16) v[i] = idx < n16 ? srcK[idx] : srcV[idx - n16];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = base + lane + 32 * i;
      if (idx < n16) dstK[idx] = v[i];
      else if (idx < 2 * n16) dstV[idx - n16] = v[i];
    }
  }
  if (d.hmk) {
    constexpr int m16 = kChunk * L::kNI * 4 / 16;   // 16-byte vectors of one side's metadata
    if (lane < 2 * m16) {
      const int side = lane / m16, idx = lane - side * m16;
      const uint4 x = reinterpret_cast<const uint4*>(side ? d.hmv : d.hmk)[idx];
      reinterpret_cast<uint4*>(slot + (side ? L::kOffMV : L::kOffMK))[idx] = x;
    }
  }
}

// HOSTOK: some pools live in host memory (see copy_host_chunk).
template <int D, bool QBF16, int FAM, bool NARROW, bool EXT, bool HOSTOK = false>
__global__ void __launch_bounds__(Warps<D, NARROW>::kThreads, Layout<D, NARROW>::kMinBlocks)
    decode_kernel(const Params p) {
  constexpr int kConsumerWarps = Warps<D, NARROW>::kConsumer;
  constexpr int kNC = Warps<D, NARROW>::kNC;
  constexpr int kChunksPerStage = Layout<D, NARROW>::kCPS;   // this layout's stage size
  using L = Layout<D, NARROW>;
  constexpr int KC = D / 16;
  constexpr int MB = D / 16;
  constexpr int DL = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + L::kStages;
  ChunkDesc* descs = reinterpret_cast<ChunkDesc*>(smem + L::kDescOff);
  int* misc = reinterpret_cast<int*>(smem + L::kMiscOff);
  volatile int* abort_flag = misc;
  uint64_t* pdone = reinterpret_cast<uint64_t*>(misc + 4);     // every producer has stopped issuing
  volatile int* slot_stage = misc + 6;                          // [kStages] last stage issued into each slot
  constexpr int kProducers = Warps<D, NARROW>::kProducers;

  // Programmatic dependent launch: the next kernel on the stream may start its
  // prologue (block-table walk and K/V prefetch) while this grid finishes; every
  // read of data a predecessor may write (q) and every global write below
  // happens after griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (p.pdl == 2) asm volatile("griddepcontrol.wait;" ::: "memory");   // nothing is read before it
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hkv = p.Hkv, G = p.G, P = p.P;
  const int cpp = P / kChunk;
  const bool sparse = p.sel_pages != nullptr;
  // A selection's entries are dealt round-robin: split s reads entries s,
  // s + S, s + 2S, ... (S = num_splits), so the splits of a row get equal
  // shares of whatever count the row has.  Dense pages: split s reads chunks
  // [s cps, (s + 1) cps).  sel_entry: the entry of this CTA's local chunk i.
  auto sel_entry = [&](int i) -> int { return (i / cpp) * p.num_splits + split; };

  // Codec and slot of logical page `page` (both -1 outside the table).
  auto lookup = [&](int page, int& codec, long long& slot) {
    codec = -1;
    slot = -1;
    if (page >= 0 && page < p.max_pages) {
      codec = p.page_codec[(size_t)b * p.max_pages + page];
      slot = p.block_table[(size_t)b * p.max_pages + page];
    }
  };
  // The producer lane's first chunk: its selection entry, or its codec and
  // slot, requested before the sequence length arrives (indices stay inside
  // their arrays whatever the length turns out to be).
  const size_t sel_row = ((size_t)b * Hkv + h) * (size_t)p.sel_width;
  int pf_page = -1, pf_codec = -1;
  long long pf_slot = -1;
  if (warp >= kConsumerWarps) {
    const int i0 = (warp - kConsumerWarps) * Warps<D, NARROW>::kBatch + lane;
    if (sparse) {
      const int v = sel_entry(i0);
      pf_page = (v < p.sel_width) ? p.sel_pages[sel_row + v] : -1;
    } else {
      pf_page = (split * p.cps + i0) / cpp;
      lookup(pf_page, pf_codec, pf_slot);
    }
  }

  int seq_len = p.seq_lens[b];
  seq_len = max(0, min(seq_len, p.max_pages * P));
  const int n_pages_b = (seq_len + P - 1) / P;
  ChunkList cl{0, 0, 0};
  const int c_begin = sparse ? 0 : split * p.cps;
  int n_local, n_active;
  if (!sparse) {
    cl = dense_chunks(seq_len, EXT ? p.window : 0, EXT ? p.sinks : 0);
    n_local = min(cl.n, c_begin + p.cps) - c_begin;
    n_active = (cl.n + p.cps - 1) / p.cps;
  } else {
    const int cnt = p.sel_count[b * Hkv + h];
    const int n_sel = max(0, min(cnt, p.sel_width));
    n_local = (n_sel > split) ? (n_sel - split + p.num_splits - 1) / p.num_splits * cpp : 0;
    n_active = min(n_sel, p.num_splits);
    if (cnt > p.sel_width && split == 0 && threadIdx.x == 0 && p.status) atomicAdd(p.status, 1u);
  }
  const size_t row0 = (size_t)b * (Hkv * G) + (size_t)h * G;  // first query head row

  if (n_local <= 0) {
    if (n_active == 0 && split == 0) {  // empty visible set: o = 0, lse2 = -inf
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const size_t o = (row0 + idx / D) * D + idx % D;
        if (p.out) {
          if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(0.f);
          else reinterpret_cast<__half*>(p.out)[o] = __float2half_rn(0.f);
        }
        if (p.out_f32) p.out_f32[o] = 0.f;
        if (p.lse2_out && idx % D == 0) p.lse2_out[row0 + idx / D] = -INFINITY;
      }
    }
    return;
  }
  const int n_stages = (n_local + kChunksPerStage - 1) / kChunksPerStage;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 2);  // producer: expect_tx arrival + descriptor arrival
      mbar_init(&empty[s], kConsumerWarps);
    }
    misc[0] = 0;  // timeout flag
    mbar_init(pdone, kProducers);
    for (int s = 0; s < L::kStages; ++s) slot_stage[s] = -1;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= kConsumerWarps) {
    // ------------------------------------------------------------ producers
    // Chunks are translated 32 at a time, one per lane; producer pw takes the
    // batches pw, pw + kProducers, ...  Lookups run one batch ahead of the
    // copies: while a batch's stages are issued, the warp's next batch's codec
    // and slot loads and the selection entries of the batch after that are in
    // flight.  The first batch's lookups were issued before the sequence
    // length was known.  (A producer's consecutive stages are never more than
    // kStages apart, so its parity waits on a slot are at most one phase ahead.)
    const int pw = warp - kConsumerWarps;
    constexpr int kBatch = Warps<D, NARROW>::kBatch;
    constexpr int kStride = kBatch * kProducers;
    static_assert(kProducers == 1 || kBatch / kChunksPerStage * (kProducers - 1) + 1 <= L::kStages,
                  "a producer's consecutive stages must stay within the ring");
    int cur_page = pf_page, cur_codec = pf_codec;
    long long cur_slot = pf_slot;
    if (sparse) {
      lookup(cur_page, cur_codec, cur_slot);
    } else if (EXT) {   // the speculative lookup assumed the unwindowed list
      cur_page = cl.chunk(c_begin + pw * kBatch + lane) / cpp;
      lookup(cur_page, cur_codec, cur_slot);
    }
    auto page_at = [&](int base) -> int {
      if (base >= n_local) return -1;
      if (!sparse) return (EXT ? cl.chunk(c_begin + base + lane) : c_begin + base + lane) / cpp;
      const int v = sel_entry(base + lane);
      return (v < p.sel_width) ? p.sel_pages[sel_row + v] : -1;
    };
    int nxt_page = page_at(pw * kBatch + kStride);
    bool stop = false;
    int withheld = -1;  // stage (warp-uniform)
    for (int base = pw * kBatch; base < n_local && !stop; base += kStride) {
      int nxt_codec = -1;
      long long nxt_slot = -1;
      if (base + kStride < n_local) lookup(nxt_page, nxt_codec, nxt_slot);
      const int nn_page = page_at(base + 2 * kStride);

      ChunkDesc d;
      d.codec = -1;
      d.vmask = 0;
      d.kscale = 1.f;
      d.vscale = 1.f;
      d.hk = d.hv = d.hmk = d.hmv = nullptr;
      uint32_t kv_bytes = 0, m_bytes = 0;
      const uint8_t *srcK = nullptr, *srcV = nullptr, *srcMK = nullptr, *srcMV = nullptr;
      if (lane < kBatch && base + lane < n_local) {
        const int ci = sparse ? sel_entry(base + lane) * cpp + (base + lane) % cpp
                              : (EXT ? cl.chunk(c_begin + base + lane) : c_begin + base + lane);
        const int cip = ci - (ci / cpp) * cpp;
        // anomalies are counted once per page: at its first listed chunk
        const bool first = cip == 0 || (EXT && !sparse && ci == cl.cw && (cl.cs == 0 || (cl.cs - 1) / cpp != ci / cpp));
        const int page = cur_page;
        bool good = true;
        if (sparse && (page < 0 || page >= n_pages_b)) {
          good = false;
          if (cip == 0 && p.status) atomicAdd(p.status, 1u);
        }
        if (good) {
          const int tok0 = page * P + cip * kChunk;
          const uint32_t vm = EXT ? chunk_rows(tok0, seq_len, p.window, p.sinks)
                                  : (uint32_t)max(0, min(kChunk, seq_len - tok0));
          if (vm != 0u) {
            const int codec = cur_codec;
            const long long slot_id = cur_slot;
            // INT2 pages are read by the extended kernels only
            bool ok = codec >= 0 && codec <= (EXT ? ARGUS_INT1_G32 : ARGUS_INT4_G32) && p.codes[codec] != nullptr;
            if (ok) {
              const int fam = codec_family(codec);
              ok = (FAM == kFamMixed) || (FAM == fam);
            }
            if (ok) ok = slot_id >= 0 && slot_id < p.n_slots[codec];
            if (NARROW && codec <= ARGUS_BF16) ok = false;   // 16-bit rows do not fit a narrow slot
            if (!ok) {
              if (first && p.status) atomicAdd(p.status, 1u);
            } else {
              const int rowb = row_bytes(codec, D);
              const size_t rk = (((size_t)slot_id * 2 + 0) * Hkv + h) * P + (size_t)cip * kChunk;
              const size_t rv = (((size_t)slot_id * 2 + 1) * Hkv + h) * P + (size_t)cip * kChunk;
              srcK = p.codes[codec] + rk * rowb;
              srcV = p.codes[codec] + rv * rowb;
              kv_bytes = kChunk * rowb;
              d.codec = codec;
              if (affine_codec(codec)) {
                srcMK = p.meta[codec] + rk * (L::kNI * 4);
                srcMV = p.meta[codec] + rv * (L::kNI * 4);
                m_bytes = kChunk * L::kNI * 4;
              }
              if (HOSTOK && ((p.host_mask >> codec) & 1u)) {   // read in place by the consumer
                d.hk = srcK;
                d.hv = srcV;
                d.hmk = srcMK;
                d.hmv = srcMV;
                kv_bytes = m_bytes = 0;
              }
              if (codec == ARGUS_FP8_E4M3 || codec == ARGUS_INT8) {
                const float* ms = reinterpret_cast<const float*>(p.meta[codec]);
                d.kscale = ms[((size_t)slot_id * 2 + 0) * Hkv + h];
                d.vscale = ms[((size_t)slot_id * 2 + 1) * Hkv + h];
              }
              d.vmask = vm;
            }
          }
        }
      }
      const uint32_t my_bytes = 2 * (kv_bytes + m_bytes);
      const int n_batch_stages = min(kBatch / kChunksPerStage, (n_local - base + kChunksPerStage - 1) / kChunksPerStage);
      for (int st = 0; st < n_batch_stages; ++st) {
        const int s = base / kChunksPerStage + st;
        const int slot = s % L::kStages;
        if (s >= L::kStages) {
          if (!mbar_wait(&empty[slot], ((s / L::kStages) - 1) & 1, reinterpret_cast<volatile uint32_t*>(misc),
                         p.wait_ns)) {
            if (lane == 0) {
              *abort_flag = 1;
              if (p.status) atomicOr(p.status, kStatusTimeoutBit);
            }
            stop = true;
            break;
          }
          if (*abort_flag) {  // the consumers gave up (they arrive on empty after setting the flag)
            stop = true;
            break;
          }
        }
        const bool mine = (lane / kChunksPerStage) == st;  // these lanes own this stage's chunks
        uint32_t total = mine ? my_bytes : 0u;
#pragma unroll
        for (int o = 1; o < kChunksPerStage; o <<= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
        total = __shfl_sync(0xffffffffu, total, kChunksPerStage * st);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], total);
        __syncwarp();
        if (mine) {
          const int j = lane % kChunksPerStage;
          if (kv_bytes) {
            uint8_t* dst = smem + slot * L::kStageBytes + j * L::kChunkBytes;
            bulk_g2s(dst + L::kOffK, srcK, kv_bytes, &full[slot]);
            bulk_g2s(dst + L::kOffV, srcV, kv_bytes, &full[slot]);
            if (m_bytes) {
              bulk_g2s(dst + L::kOffMK, srcMK, m_bytes, &full[slot]);
              bulk_g2s(dst + L::kOffMV, srcMV, m_bytes, &full[slot]);
            }
          }
          descs[slot * kChunksPerStage + j] = d;
        }
        __syncwarp();
        if (lane == 0) slot_stage[slot] = s;
        if (s == p.stall_stage) withheld = s;
        else if (lane == 0) mbar_arrive(&full[slot]);
      }
      cur_page = nxt_page;
      cur_codec = nxt_codec;
      cur_slot = nxt_slot;
      nxt_page = nn_page;
    }
    // Wind-down.  A producer that withheld an arrival completes it once the
    // consumers have given up on that stage; every producer then reports
    // that it stopped issuing (after a timeout the consumers drain the ring
    // before reusing it).  Every wait here is bounded as well.
    if (withheld >= 0) {
      const unsigned long long t0 = global_ns();
      // the consumers start their wait on this stage within microseconds of
      // its issue; twice their limit leaves ample margin
      while (!*abort_flag && global_ns() - t0 <= 2 * p.wait_ns) __nanosleep(1000);
      if (lane == 0) mbar_arrive(&full[withheld % L::kStages]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(pdone);
    return;
  }

  // -------------------------------------------------------------- consumers
  if (warp == 0 && lane < G) {
    // pull this CTA's query rows toward L2 while the predecessor finishes
    const char* qrow = reinterpret_cast<const char*>(p.q) + ((row0 + lane) * D) * 2;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow));
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int r = lane >> 2, t = lane & 3;
  // query fragments (B operand of Q.K: k = head_dim, n = query head r)
  uint32_t qf[KC][2], qb[KC][2];
  uint32_t qf8[KC][2];  // qf in the byte-codec dim order (see load_k_frags)
  float qgs[D / 32][2];  // per-group query sums of heads 2t, 2t+1 (fp16 domain)
  float qscale_h0 = 1.f, qscale_h1 = 1.f;  // 2^-e of heads 2t, 2t+1 (bf16 q in fp16 MMAs)
  {
    float qv[D / 4];
    const bool live = r < G;
    // every query load of this lane is issued here, in one round trip: the
    // run layout (x32) and the byte-codec layout (x64)
    uint4 x32[D / 32], x64[D / 64][2];
    {
      const uint16_t* qrow = reinterpret_cast<const uint16_t*>(p.q) + (row0 + r) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i)
        x32[i] = live ? *reinterpret_cast<const uint4*>(qrow + 32 * i + 8 * t) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < D / 64; ++j) {
        const bool need = live && FAM != kFamBF16;
        x64[j][0] = need ? *reinterpret_cast<const uint4*>(qrow + 64 * j + 16 * t) : make_uint4(0, 0, 0, 0);
        x64[j][1] = need ? *reinterpret_cast<const uint4*>(qrow + 64 * j + 16 * t + 8) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const uint4 x = x32[i];
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint16_t bits = (wv[e / 2] >> (16 * (e & 1))) & 0xFFFFu;
        qv[8 * i + e] = QBF16 ? __uint_as_float((uint32_t)bits << 16)
                              : __half2float(__ushort_as_half(bits));
      }
      if (FAM != kFamF16) {
        qb[2 * i][0] = prmt(x.x, x.z, 0x5410);
        qb[2 * i][1] = prmt(x.x, x.z, 0x7632);
        qb[2 * i + 1][0] = prmt(x.y, x.w, 0x5410);
        qb[2 * i + 1][1] = prmt(x.y, x.w, 0x7632);
      }
    }
    if (FAM != kFamBF16) {
      float e_scale = 1.f;  // power of two bringing max|q| of this head into [2^14, 2^15)
      if (QBF16) {
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < D / 4; ++e) mx = fmaxf(mx, fabsf(qv[e]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        int ex = 0;
        if (mx > 0.f) ex = 14 - ilogbf(mx);
        ex = max(-100, min(100, ex));
        e_scale = ldexpf(1.f, ex);
        const float inv = ldexpf(1.f, -ex);
        qscale_h0 = __shfl_sync(0xffffffffu, inv, 4 * (2 * t));
        qscale_h1 = __shfl_sync(0xffffffffu, inv, 4 * (2 * t + 1));
      }
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        const float* e8 = qv + 8 * i;
        qf[2 * i][0] = pack_f16x2(e8[0] * e_scale, e8[4] * e_scale);
        qf[2 * i][1] = pack_f16x2(e8[1] * e_scale, e8[5] * e_scale);
        qf[2 * i + 1][0] = pack_f16x2(e8[2] * e_scale, e8[6] * e_scale);
        qf[2 * i + 1][1] = pack_f16x2(e8[3] * e_scale, e8[7] * e_scale);
        // sum of this head's fp16 query values over 32-dim group i (INT4 zero-points)
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) part += __half2float(__float2half_rn(e8[e] * e_scale));
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        qgs[i][0] = __shfl_sync(0xffffffffu, part, 4 * (2 * t));
        qgs[i][1] = __shfl_sync(0xffffffffu, part, 4 * (2 * t + 1));
      }
      // the same query values (same fp16 rounding) in the byte-codec order
#pragma unroll
      for (int j = 0; j < D / 64; ++j) {
        const uint4* x = x64[j];
        const uint32_t wv[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
        float e16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint16_t bits = (wv[e / 2] >> (16 * (e & 1))) & 0xFFFFu;
          e16[e] = (QBF16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits))) * e_scale;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          qf8[4 * j + cc][0] = pack_f16x2(e16[4 * cc], e16[4 * cc + 1]);
          qf8[4 * j + cc][1] = pack_f16x2(e16[4 * cc + 2], e16[4 * cc + 3]);
        }
      }
    }
  }

  float acc[MB][4];
#pragma unroll
  for (int j = 0; j < MB; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  // running max (log2 domain) and lane-partial sums of heads 2t, 2t+1; the
  // accumulator is kept in units of sigma (the largest V scale seen so far)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, sigma = 0.f;
  bool alive = true;

  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % L::kStages;
    if (alive && !mbar_wait(&full[slot], (s / L::kStages) & 1, reinterpret_cast<volatile uint32_t*>(misc),
                            p.wait_ns)) {
      alive = false;
      if (lane == 0) {
        *abort_flag = 1;
        if (p.status) atomicOr(p.status, kStatusTimeoutBit);
      }
    }
    if (alive && *abort_flag) alive = false;
    ChunkDesc dsc[kNC];
    const uint8_t* cptr[kNC];
    bool any = false;
#pragma unroll
    for (int c = 0; c < kNC; ++c) {
      dsc[c] = descs[slot * kChunksPerStage + warp * kNC + c];
      cptr[c] = smem + slot * L::kStageBytes + (warp * kNC + c) * L::kChunkBytes;
      any |= dsc[c].codec >= 0;
    }
    if constexpr (HOSTOK) {
      if (alive) {
#pragma unroll
        for (int c = 0; c < kNC; ++c)
          if (dsc[c].codec >= 0 && dsc[c].hk) copy_host_chunk<D, NARROW>(dsc[c], const_cast<uint8_t*>(cptr[c]), lane);
        __syncwarp();
      }
    }
    if (alive && any) {
      // ---- scores S^T[token][head] = K . q; a group whose chunks share one
      // codec runs as straight-line code so that all MMAs overlap
      float sv[kNC][4];
      const bool same = (kNC == 2) && (dsc[0].codec >= 0) && (dsc[kNC - 1].codec == dsc[0].codec);
      const float fq0 = qscale_h0, fq1 = qscale_h1;
      auto scores = [&](int codec, int c0, int ncg) {
        const uint8_t* const* cp = cptr + c0;
        const ChunkDesc* dd = dsc + c0;
        if constexpr (kNC == 2) {
          if (ncg == 2) {
            switch (codec) {
              case ARGUS_FP16: group_scores<D, ARGUS_FP16, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
              case ARGUS_BF16: group_scores<D, ARGUS_BF16, 2, true, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, 1.f, 1.f, p.scale_log2, sv, c0); break;
              case ARGUS_FP8_E4M3: group_scores<D, ARGUS_FP8_E4M3, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
              case ARGUS_INT8: group_scores<D, ARGUS_INT8, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
              default:
                if constexpr (EXT) {   // the INT2 tier exists in the extended kernels only
                  if (codec == ARGUS_INT2_G32) {
                    group_scores<D, ARGUS_INT2_G32, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
                    break;
                  }
                  if (codec == ARGUS_INT1_G32) {
                    group_scores<D, ARGUS_INT1_G32, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
                    break;
                  }
                }
                group_scores<D, ARGUS_INT4_G32, 2, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
                break;
            }
            return;
          }
        }
        switch (codec) {
          case ARGUS_FP16: group_scores<D, ARGUS_FP16, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
          case ARGUS_BF16: group_scores<D, ARGUS_BF16, 1, true, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, 1.f, 1.f, p.scale_log2, sv, c0); break;
          case ARGUS_FP8_E4M3: group_scores<D, ARGUS_FP8_E4M3, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
          case ARGUS_INT8: group_scores<D, ARGUS_INT8, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0); break;
          default:
            if constexpr (EXT) {   // the INT2 tier exists in the extended kernels only
              if (codec == ARGUS_INT2_G32) {
                group_scores<D, ARGUS_INT2_G32, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
                break;
              }
              if (codec == ARGUS_INT1_G32) {
                group_scores<D, ARGUS_INT1_G32, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
                break;
              }
            }
            group_scores<D, ARGUS_INT4_G32, 1, false, NARROW, EXT>(cp, dd, r, t, qf, qb, qf8, qgs, fq0, fq1, p.scale_log2, sv, c0);
            break;
        }
      };
      if (same) {
        scores(dsc[0].codec, 0, 2);
      } else {
#pragma unroll
        for (int c = 0; c < kNC; ++c) {
          sv[c][0] = sv[c][1] = sv[c][2] = sv[c][3] = -INFINITY;
          if (dsc[c].codec >= 0) scores(dsc[c].codec, c, 1);
        }
      }
      // ---- one online-softmax update for all chunks of the group
      float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
      for (int c = 0; c < kNC; ++c) {
        t0 = fmaxf(t0, fmaxf(sv[c][0], sv[c][2]));
        t1 = fmaxf(t1, fmaxf(sv[c][1], sv[c][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
      }
      // the new maxima are finite: token 0 of a non-empty chunk is visible
      const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      // V scales: codecs without one count as 1; sigma only grows, so every
      // chunk's weight vs / sigma is <= 1 and P stays in [0, 1] before the MMA
      float vmax = sigma;
#pragma unroll
      for (int c = 0; c < kNC; ++c)
        if (dsc[c].codec >= 0 && dsc[c].vscale > 0.f) vmax = fmaxf(vmax, dsc[c].vscale);
      float gs = 1.f;
      if (vmax > sigma) {
        gs = (sigma > 0.f) ? sigma / vmax : 0.f;
        sigma = vmax;
      }
      const float g0 = al0 * gs, g1 = al1 * gs;
      if (__any_sync(0xffffffffu, g0 != 1.f || g1 != 1.f)) {  // most chunks move neither max nor sigma
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          acc[j][0] *= g0;
          acc[j][1] *= g1;
          acc[j][2] *= g0;
          acc[j][3] *= g1;
        }
      }
      float pw[kNC][4];
      bool skip[kNC];
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int c = 0; c < kNC; ++c) {
        const float p0 = fast_exp2(sv[c][0] - mn0), p1 = fast_exp2(sv[c][1] - mn1);
        const float p2 = fast_exp2(sv[c][2] - mn0), p3 = fast_exp2(sv[c][3] - mn1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // all-zero V codes (scale 0) and empty slots contribute nothing
        skip[c] = !(dsc[c].codec >= 0 && dsc[c].vscale > 0.f);
        const float w = skip[c] ? 0.f : dsc[c].vscale / sigma;
        pw[c][0] = p0 * w;
        pw[c][1] = p1 * w;
        pw[c][2] = p2 * w;
        pw[c][3] = p3 * w;
      }
      // ---- O^T[dim][head] += V^T . (w P)^T
      auto pv = [&](int codec, int c0, int ncg) {
        const uint8_t* const* cp = cptr + c0;
        if constexpr (kNC == 2) {
          if (ncg == 2) {
            switch (codec) {
              case ARGUS_FP16: group_pv<D, ARGUS_FP16, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
              case ARGUS_BF16: group_pv<D, ARGUS_BF16, 2, true, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
              case ARGUS_FP8_E4M3: group_pv<D, ARGUS_FP8_E4M3, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
              case ARGUS_INT8: group_pv<D, ARGUS_INT8, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
              default:
                if constexpr (EXT) {
                  if (codec == ARGUS_INT2_G32) {
                    group_pv<D, ARGUS_INT2_G32, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
                    break;
                  }
                  if (codec == ARGUS_INT1_G32) {
                    group_pv<D, ARGUS_INT1_G32, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
                    break;
                  }
                }
                group_pv<D, ARGUS_INT4_G32, 2, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
                break;
            }
            return;
          }
        }
        switch (codec) {
          case ARGUS_FP16: group_pv<D, ARGUS_FP16, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
          case ARGUS_BF16: group_pv<D, ARGUS_BF16, 1, true, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
          case ARGUS_FP8_E4M3: group_pv<D, ARGUS_FP8_E4M3, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
          case ARGUS_INT8: group_pv<D, ARGUS_INT8, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc); break;
          default:
            if constexpr (EXT) {
              if (codec == ARGUS_INT2_G32) {
                group_pv<D, ARGUS_INT2_G32, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
                break;
              }
              if (codec == ARGUS_INT1_G32) {
                group_pv<D, ARGUS_INT1_G32, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
                break;
              }
            }
            group_pv<D, ARGUS_INT4_G32, 1, false, NARROW>(cp, r, t, pw + c0, skip + c0, acc);
            break;
        }
      };
      if (same) {
        pv(dsc[0].codec, 0, 2);
      } else {
#pragma unroll
        for (int c = 0; c < kNC; ++c)
          if (!skip[c]) pv(dsc[c].codec, c, 1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // ------------------------------------------------- merge the consumer warps
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (sigma == 0.f) sigma = 1.f;  // nothing accumulated
  // After a timeout the ring may still be receiving copies: once every
  // producer has stopped issuing, wait (bounded) until the last stage issued
  // into each slot has received all its bytes.  Every warp sees the flag
  // here: no warp completes all its stages once another has given up.
  if (*abort_flag) {
    mbar_wait(pdone, 0, nullptr, 3 * p.wait_ns);
    for (int sl = 0; sl < L::kStages; ++sl) {
      const int x = slot_stage[sl];
      if (x >= 0) mbar_wait(&full[sl], (x / L::kStages) & 1, nullptr, 3 * p.wait_ns);
    }
  }
  consumer_bar<kConsumerWarps>();  // every warp is done with the stage ring; reuse it
  float* red_o = reinterpret_cast<float*>(smem);               // [warps][8][D]
  float* red_ml = red_o + kConsumerWarps * kMaxG * D;          // [warps][8][2]
#pragma unroll
  for (int j = 0; j < MB; ++j) {
    const int d0 = DL * r + 2 * j, d1 = d0 + 1;
    red_o[(warp * kMaxG + 2 * t) * D + d0] = acc[j][0] * sigma;
    red_o[(warp * kMaxG + 2 * t + 1) * D + d0] = acc[j][1] * sigma;
    red_o[(warp * kMaxG + 2 * t) * D + d1] = acc[j][2] * sigma;
    red_o[(warp * kMaxG + 2 * t + 1) * D + d1] = acc[j][3] * sigma;
  }
  if (r == 0) {
    red_ml[(warp * kMaxG + 2 * t) * 2 + 0] = m0;
    red_ml[(warp * kMaxG + 2 * t) * 2 + 1] = l0;
    red_ml[(warp * kMaxG + 2 * t + 1) * 2 + 0] = m1;
    red_ml[(warp * kMaxG + 2 * t + 1) * 2 + 1] = l1;
  }
  consumer_bar<kConsumerWarps>();
  // one float4 of one head per thread (G * D / 4 <= consumer threads): each
  // thread forms its head's merge weights itself, so no further barrier
  static_assert(kMaxG * D / 4 <= kConsumerWarps * 32, "one float4 per consumer thread");
  const int tid = threadIdx.x;
  const int g = tid / (D / 4), c4 = tid - g * (D / 4);
  if (g < G) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_ml[(w * kMaxG + g) * 2]);
    float Lsum = 0.f;
    float f[kConsumerWarps];
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      f[w] = (M == -INFINITY) ? 0.f : fast_exp2(red_ml[(w * kMaxG + g) * 2] - M);
      Lsum += red_ml[(w * kMaxG + g) * 2 + 1] * f[w];
    }
    const float inv = (Lsum > 0.f) ? 1.f / Lsum : 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(red_o + (w * kMaxG + g) * D + 4 * c4);
      const float fw = f[w] * inv;
      o.x += fw * x.x;
      o.y += fw * x.y;
      o.z += fw * x.z;
      o.w += fw * x.w;
    }
    const float lse2 = (Lsum > 0.f) ? M + log2f(Lsum) : -INFINITY;
    if (n_active == 1) {
      const size_t oi = (row0 + g) * D + 4 * c4;
      if (p.out) {
        uint2 v2;
        if (p.out_bf16) {
          v2.x = pack_bf16x2(o.x, o.y);
          v2.y = pack_bf16x2(o.z, o.w);
        } else {
          v2.x = pack_f16x2(o.x, o.y);
          v2.y = pack_f16x2(o.z, o.w);
        }
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + oi) = v2;
      }
      if (p.out_f32) *reinterpret_cast<float4*>(p.out_f32 + oi) = o;
      if (p.lse2_out && c4 == 0) p.lse2_out[row0 + g] = lse2;
    } else {
      const size_t bh = (size_t)b * Hkv + h;
      float* po = p.part_o + (bh * p.num_splits + split) * G * D + (size_t)g * D + 4 * c4;
      *reinterpret_cast<float4*>(po) = o;
      if (c4 == 0) p.part_lse[(bh * p.num_splits + split) * G + g] = lse2;
    }
  }
}

// Split combine: one CTA per (batch row, query head).  Launched after the
// decode grid with programmatic dependent launch, it waits for the partials,
// then every thread loads its share of (split, 16-byte column) partials at once
// and the CTA folds them by log2-sum-exp.  Rows with at most one active split
// were written by the decode kernel itself.
template <int D>
__global__ void __launch_bounds__(kFoldThreads) decode_fold_kernel(const Params p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int D4 = D / 4;
  constexpr int GROUPS = kFoldThreads / D4;     // split groups per column
  __shared__ float4 sh_acc[GROUPS][D4];
  const int hq = blockIdx.x, b = blockIdx.y;
  const int G = p.G, Hkv = p.Hkv;
  const int h = hq / G, g = hq - h * G;
  int seq_len = p.seq_lens[b];
  seq_len = max(0, min(seq_len, p.max_pages * p.P));
  int n_active;
  if (!p.sel_pages) n_active = (dense_chunks(seq_len, p.window, p.sinks).n + p.cps - 1) / p.cps;
  else n_active = min(max(0, min(p.sel_count[b * Hkv + h], p.sel_width)), p.num_splits);
  if (n_active <= 1) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t bh = (size_t)b * Hkv + h;
  const float* po = p.part_o + bh * p.num_splits * G * D + (size_t)g * D;
  const float* pl = p.part_lse + bh * p.num_splits * G + g;
  const int tid = threadIdx.x;
  const int col = tid % D4, grp = tid / D4;
  // each thread folds splits grp, grp + GROUPS, ... of one 16-byte column,
  // kKPT of them per batch with every load of the batch issued first, keeping
  // its own running (max, sum, vector) in the log2 domain
  constexpr int kKPT = 8;
  float m = -INFINITY, l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < n_active; base += kKPT * GROUPS) {
    float4 x[kKPT];
    float ls[kKPT];
#pragma unroll
    for (int k = 0; k < kKPT; ++k) {
      const int s2 = base + grp + k * GROUPS;
      if (s2 < n_active) {
        x[k] = __ldcg(reinterpret_cast<const float4*>(po + (size_t)s2 * G * D) + col);
        ls[k] = __ldcg(pl + (size_t)s2 * G);
      } else {
        x[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        ls[k] = -INFINITY;
      }
    }
    float bm = m;
#pragma unroll
    for (int k = 0; k < kKPT; ++k) bm = fmaxf(bm, ls[k]);
    if (bm == -INFINITY) continue;
    const float r0 = fast_exp2(m - bm);
    a.x *= r0; a.y *= r0; a.z *= r0; a.w *= r0;
    l *= r0;
#pragma unroll
    for (int k = 0; k < kKPT; ++k) {
      const float w = fast_exp2(ls[k] - bm);
      a.x += w * x[k].x;
      a.y += w * x[k].y;
      a.z += w * x[k].z;
      a.w += w * x[k].w;
      l += w;
    }
    m = bm;
  }
  // combine the GROUPS partial folds of each column
  __shared__ float sh_m[GROUPS][D4];
  __shared__ float sh_l[GROUPS][D4];
  sh_m[grp][col] = m;
  sh_l[grp][col] = l;
  sh_acc[grp][col] = a;
  __syncthreads();
  if (grp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < GROUPS; ++q) M = fmaxf(M, sh_m[q][col]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int q = 0; q < GROUPS; ++q) {
        const float w = fast_exp2(sh_m[q][col] - M);
        L += w * sh_l[q][col];
        o.x += w * sh_acc[q][col].x;
        o.y += w * sh_acc[q][col].y;
        o.z += w * sh_acc[q][col].z;
        o.w += w * sh_acc[q][col].w;
      }
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    const float ov[4] = {o.x * inv, o.y * inv, o.z * inv, o.w * inv};
    const size_t row = (size_t)b * Hkv * G + hq;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const size_t oi = row * D + 4 * col + e;
      if (p.out) {
        if (p.out_bf16) reinterpret_cast<__nv_bfloat16*>(p.out)[oi] = __float2bfloat16_rn(ov[e]);
        else reinterpret_cast<__half*>(p.out)[oi] = __float2half_rn(ov[e]);
      }
      if (p.out_f32) p.out_f32[oi] = ov[e];
    }
    if (p.lse2_out && col == 0) p.lse2_out[row] = (L > 0.f) ? M + log2f(L) : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct Plan {
  int D, G, cps, num_splits, fam;
  bool q_bf16, narrow;
  bool ext;   // extended kernels: a sliding window or an INT2 pool
  bool host;  // some pool lives in host memory
  size_t part_o_bytes, ws_bytes;
};

static argus_status plan(const argus_decode_args* a, Plan* pl) {
  if (!a) return fail(ARGUS_E_INVALID, "decode: args is NULL");
  const argus_geom& g = a->g;
  if (g.n_q_heads <= 0 || g.n_kv_heads <= 0 || g.head_dim <= 0 || g.page_tokens <= 0)
    return fail(ARGUS_E_INVALID, "decode: geometry fields must be positive");
  if (g.n_q_heads % g.n_kv_heads != 0)
    return fail(ARGUS_E_INVALID, "decode: n_q_heads %% n_kv_heads != 0");
  const int G = g.n_q_heads / g.n_kv_heads;
  if (G > kMaxG) return fail(ARGUS_E_UNSUPPORTED, "decode: G = %d > 8 query heads per KV head", G);
  if (a->pdl < 0 || a->pdl > 2) return fail(ARGUS_E_INVALID, "decode: pdl must be 0, 1 or 2");
  if (g.head_dim != 64 && g.head_dim != 128)
    return fail(ARGUS_E_UNSUPPORTED, "decode: head_dim %d (supported: 64, 128)", g.head_dim);
  if (g.page_tokens % kChunk != 0)
    return fail(ARGUS_E_UNSUPPORTED, "decode: page_tokens %d is not a multiple of 16", g.page_tokens);
  if (a->batch < 0) return fail(ARGUS_E_INVALID, "decode: negative batch");
  if (a->batch > 65535 || g.n_kv_heads > 65535) return fail(ARGUS_E_UNSUPPORTED, "decode: batch or n_kv_heads too large");
  if (a->q_dtype != ARGUS_FP16 && a->q_dtype != ARGUS_BF16)
    return fail(ARGUS_E_INVALID, "decode: q_dtype must be FP16 or BF16");
  if (a->max_pages <= 0) return fail(ARGUS_E_INVALID, "decode: max_pages must be positive");
  if ((long long)a->max_pages * g.page_tokens > (1LL << 30))
    return fail(ARGUS_E_UNSUPPORTED, "decode: max_pages * page_tokens too large");
  if ((a->sel_pages == nullptr) != (a->sel_count == nullptr))
    return fail(ARGUS_E_INVALID, "decode: sel_pages and sel_count must both be set or both NULL");
  if (a->sel_pages && a->sel_width <= 0) return fail(ARGUS_E_INVALID, "decode: sel_width must be positive");
  if (a->n_pools < 0 || a->n_pools > kNumCodecs || (a->n_pools > 0 && !a->pools))
    return fail(ARGUS_E_INVALID, "decode: bad pool list");
  if (!std::isfinite(a->softmax_scale)) return fail(ARGUS_E_INVALID, "decode: softmax_scale not finite");
  if (a->out && a->out_dtype != ARGUS_FP16 && a->out_dtype != ARGUS_BF16)
    return fail(ARGUS_E_INVALID, "decode: out_dtype must be FP16 or BF16");
  bool seen[kNumCodecs] = {};
  bool has_bf16 = false, has_f16 = false;
  for (int i = 0; i < a->n_pools; ++i) {
    const argus_pool& pool = a->pools[i];
    if (pool.codec < 0 || pool.codec > ARGUS_INT1_G32) return fail(ARGUS_E_INVALID, "decode: pool %d has codec %d", i, pool.codec);
    if (pool.placement != ARGUS_PLACE_DEVICE && pool.placement != ARGUS_PLACE_HOST)
      return fail(ARGUS_E_INVALID, "decode: pool %d has placement %d", i, pool.placement);
    if (seen[pool.codec]) return fail(ARGUS_E_INVALID, "decode: two pools with codec %d", pool.codec);
    seen[pool.codec] = true;
    if (pool.n_slots < 0) return fail(ARGUS_E_INVALID, "decode: pool %d n_slots < 0", i);
    if (pool.n_slots > 0) {
      if (!pool.codes || (reinterpret_cast<uintptr_t>(pool.codes) & 15))
        return fail(ARGUS_E_INVALID, "decode: pool %d codes NULL or not 16-byte aligned", i);
      if (pool.codec >= ARGUS_FP8_E4M3 &&
          (!pool.meta || (reinterpret_cast<uintptr_t>(pool.meta) & 15)))
        return fail(ARGUS_E_INVALID, "decode: pool %d meta NULL or not 16-byte aligned", i);
    }
    if (pool.codec == ARGUS_BF16) has_bf16 = true;
    else has_f16 = true;
  }
  pl->q_bf16 = (a->q_dtype == ARGUS_BF16);
  if (has_bf16 && !pl->q_bf16)
    return fail(ARGUS_E_UNSUPPORTED, "decode: BF16 pages need a BF16 query");
  pl->fam = (has_bf16 && has_f16) ? kFamMixed : (has_bf16 ? kFamBF16 : kFamF16);
  pl->D = g.head_dim;
  pl->G = G;
  // extended kernels: a sliding window, INT2 or INT1 pages
  pl->ext = a->window_tokens > 0 || seen[ARGUS_INT2_G32] || seen[ARGUS_INT1_G32];
  pl->host = false;
  for (int i = 0; i < a->n_pools; ++i) pl->host |= a->pools[i].placement == ARGUS_PLACE_HOST;
  if (pl->host && pl->ext)
    return fail(ARGUS_E_UNSUPPORTED, "decode: host-memory pools with a sliding window or an INT2 / INT1 pool");
  // narrow ring: every pool holds byte or sub-byte codes, head_dim 128
  pl->narrow = g.head_dim == 128 && !has_bf16 && !seen[ARGUS_FP16] && a->n_pools > 0 && !pl->host;
  const long long cps_unit = pl->narrow ? chunks_per_stage<true>() : kChunksPerStage;
  const int cpp = g.page_tokens / kChunk;
  if (a->window_tokens < 0 || a->sink_tokens < 0)
    return fail(ARGUS_E_INVALID, "decode: window_tokens and sink_tokens must be >= 0");
  if (a->window_tokens > 0 && a->sel_pages)
    return fail(ARGUS_E_UNSUPPORTED, "decode: a sliding window applies to dense pages, not to a selection");
  long long max_chunks = a->sel_pages ? (long long)a->sel_width * cpp : (long long)a->max_pages * cpp;
  if (a->window_tokens > 0)   // sink chunks + window chunks (+1 when the window starts mid-chunk)
    max_chunks = std::min<long long>(max_chunks, ((long long)a->sink_tokens + kChunk - 1) / kChunk +
                                                     ((long long)a->window_tokens + kChunk - 1) / kChunk + 1);
  const long long rows = (long long)std::max(a->batch, 1) * g.n_kv_heads;
  const long long slots = (long long)device_sm_count() * (g.head_dim == 64 ? 2 : 1);
  if (a->sel_pages) {
    // Selected pages are dealt round-robin over the splits, so every split of
    // a row gets an equal share of its actual count, whatever part of the
    // width it uses.  Each split is a CTA that pays the whole lookup-and-load
    // latency: automatically, one wave (one CTA per resident slot).
    long long ns = a->num_splits > 0 ? a->num_splits : std::max<long long>(1, slots / rows);
    ns = std::min<long long>({ns, (long long)a->sel_width, (long long)kMaxSplits});
    pl->num_splits = (int)std::max<long long>(1, ns);
    pl->cps = (int)max_chunks;   // unused by a selection
  } else {
    long long cps;
    if (a->num_splits > 0) {
      cps = (max_chunks + a->num_splits - 1) / a->num_splits;
    } else {
      // About ten CTAs per SM, so that rows of unequal length balance.  A
      // sliding window gives every row the same bounded work: one wave of
      // CTAs (about one per SM) beats ten short ones per SM there.
      const long long total = rows * max_chunks;
      const long long target = (a->window_tokens > 0 ? 1LL : 10LL) * device_sm_count();
      cps = std::max<long long>(cps_unit, (total + target - 1) / target);
    }
    cps = std::max<long long>(cps, (max_chunks + kMaxSplits - 1) / kMaxSplits);
    cps = std::max<long long>(cps_unit, (cps + cps_unit - 1) / cps_unit * cps_unit);
    pl->cps = (int)cps;
    pl->num_splits = (int)std::max<long long>(1, (max_chunks + cps - 1) / cps);
  }
  if (pl->num_splits > 65535) return fail(ARGUS_E_UNSUPPORTED, "decode: too many splits");
  pl->part_o_bytes = (size_t)std::max(a->batch, 1) * g.n_kv_heads * pl->num_splits * G * g.head_dim * 4;
  pl->ws_bytes = pl->part_o_bytes +
                 (size_t)std::max(a->batch, 1) * g.n_kv_heads * pl->num_splits * G * 4;
  return ARGUS_OK;
}

template <int D, bool QBF16, int FAM, bool NARROW, bool EXT, bool HOSTOK = false>
static argus_status launch_t(const Params& p, dim3 grid, cudaStream_t s) {
  using L = Layout<D, NARROW>;
  static PerContext configured;
  argus_status st = configured.ensure([](int) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, QBF16, FAM, NARROW, EXT, HOSTOK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "decode: smem attribute: %s", cudaGetErrorString(e));
    return ARGUS_OK;
  });
  if (st != ARGUS_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Warps<D, NARROW>::kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<D, QBF16, FAM, NARROW, EXT, HOSTOK>, p);
  if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "argus_paged_decode_attn: %s", cudaGetErrorString(e));
  if (p.num_splits > 1) {
    cudaLaunchConfig_t fc = cfg;
    fc.gridDim = dim3(p.Hkv * p.G, p.B);
    fc.blockDim = dim3(kFoldThreads);
    fc.dynamicSmemBytes = 0;
    fc.attrs = attr;  // the combine always overlaps its decode grid's tail
    fc.numAttrs = 1;
    e = cudaLaunchKernelEx(&fc, decode_fold_kernel<D>, p);
    if (e != cudaSuccess) return fail(ARGUS_E_LAUNCH, "argus_paged_decode_attn (combine): %s", cudaGetErrorString(e));
  }
  return launch_status("argus_paged_decode_attn");
}

template <int D>
static argus_status launch_d(const Params& p, const Plan& pl, dim3 grid, cudaStream_t s) {
  if (pl.host) {   // pools in host memory: the wide ring, one kernel per query type
    if (!pl.q_bf16) return launch_t<D, false, kFamMixed, false, false, true>(p, grid, s);
    return launch_t<D, true, kFamMixed, false, false, true>(p, grid, s);
  }
  if (pl.ext) {   // sliding window or INT2 / INT1 pages: one kernel per ring and query type
    if constexpr (D == 128) {
      if (pl.narrow) {
        if (!pl.q_bf16) return launch_t<D, false, kFamF16, true, true>(p, grid, s);
        return launch_t<D, true, kFamF16, true, true>(p, grid, s);
      }
    }
    if (!pl.q_bf16) return launch_t<D, false, kFamF16, false, true>(p, grid, s);
    return launch_t<D, true, kFamMixed, false, true>(p, grid, s);
  }
  if constexpr (D == 128) {
    if (pl.narrow) {
      if (!pl.q_bf16) return launch_t<D, false, kFamF16, true, false>(p, grid, s);
      return launch_t<D, true, kFamF16, true, false>(p, grid, s);
    }
  }
  if (!pl.q_bf16) return launch_t<D, false, kFamF16, false, false>(p, grid, s);
  if (pl.fam == kFamF16) return launch_t<D, true, kFamF16, false, false>(p, grid, s);
  if (pl.fam == kFamBF16) return launch_t<D, true, kFamBF16, false, false>(p, grid, s);
  return launch_t<D, true, kFamMixed, false, false>(p, grid, s);
}

}  // namespace decode
}  // namespace argus

using namespace argus;
using namespace argus::decode;

extern "C" argus_status argus_decode_workspace_bytes(const argus_decode_args* args, size_t* bytes) {
  if (!bytes) return fail(ARGUS_E_INVALID, "decode: bytes is NULL");
  Plan pl;
  argus_status st = plan(args, &pl);
  if (st != ARGUS_OK) return st;
  *bytes = pl.ws_bytes;
  return ARGUS_OK;
}

static argus_status check_io(const argus_decode_args* a) {
  if (!a->q || !a->page_codec || !a->block_table || !a->seq_lens)
    return fail(ARGUS_E_INVALID, "decode: q, page_codec, block_table and seq_lens are required");
  if (reinterpret_cast<uintptr_t>(a->q) & 15) return fail(ARGUS_E_INVALID, "decode: q not 16-byte aligned");
  if (!a->out && !a->out_f32 && !a->lse2_out) return fail(ARGUS_E_INVALID, "decode: no output given");
  if ((reinterpret_cast<uintptr_t>(a->out) & 7) || (reinterpret_cast<uintptr_t>(a->out_f32) & 15))
    return fail(ARGUS_E_INVALID, "decode: out must be 8-byte and out_f32 16-byte aligned");
  return ARGUS_OK;
}

// Fill the kernel parameters and launch; ws holds pl.ws_bytes bytes.
static argus_status run(const argus_decode_args* a, const Plan& pl, void* ws, void* stream,
                        unsigned long long wait_ns = kWaitLimitNs, int stall_stage = -1) {
  Params p{};
  p.B = a->batch;
  p.Hkv = a->g.n_kv_heads;
  p.G = pl.G;
  p.P = a->g.page_tokens;
  p.max_pages = a->max_pages;
  p.q = a->q;
  for (int c = 0; c < kNumCodecs; ++c) {
    p.codes[c] = nullptr;
    p.meta[c] = nullptr;
    p.n_slots[c] = 0;
  }
  p.host_mask = 0;
  for (int i = 0; i < a->n_pools; ++i) {
    const argus_pool& pool = a->pools[i];
    p.codes[pool.codec] = static_cast<const uint8_t*>(pool.codes);
    p.meta[pool.codec] = static_cast<const uint8_t*>(pool.meta);
    p.n_slots[pool.codec] = pool.n_slots;
    if (pool.placement == ARGUS_PLACE_HOST) {   // page-locked host memory: the device's address of it
      const void* dc = nullptr;
      const void* dm = nullptr;
      const argus_status st = pool_device_ptrs(pool, &dc, &dm);
      if (st != ARGUS_OK) return st;
      p.codes[pool.codec] = static_cast<const uint8_t*>(dc);
      p.meta[pool.codec] = static_cast<const uint8_t*>(dm);
      p.host_mask |= 1u << pool.codec;
    }
  }
  p.page_codec = a->page_codec;
  p.block_table = a->block_table;
  p.seq_lens = a->seq_lens;
  p.sel_pages = a->sel_pages;
  p.sel_count = a->sel_count;
  p.sel_width = a->sel_width;
  p.scale_log2 = a->softmax_scale * 1.4426950408889634f;
  p.out = a->out;
  p.out_bf16 = (a->out_dtype == ARGUS_BF16);
  p.out_f32 = a->out_f32;
  p.lse2_out = a->lse2_out;
  p.status = a->status;
  p.cps = pl.cps;
  p.num_splits = pl.num_splits;
  p.pdl = a->pdl;
  // at most 2^30 tokens are ever visible (max_pages * page_tokens <= 2^30):
  // larger values mean the same and keep the device arithmetic in range
  p.window = std::min(a->window_tokens, 1 << 30);
  p.sinks = a->window_tokens > 0 ? std::min(a->sink_tokens, 1 << 30) : 0;
  p.part_o = static_cast<float*>(ws);
  p.part_lse = ws ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_o_bytes) : nullptr;
  p.wait_ns = wait_ns;
  p.stall_stage = stall_stage;
  dim3 grid(pl.num_splits, a->g.n_kv_heads, a->batch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pl.D == 64) return launch_d<64>(p, pl, grid, s);
  return launch_d<128>(p, pl, grid, s);
}

static argus_status check_ws(const Plan& pl, void* ws, size_t ws_bytes) {
  if (ws_bytes < pl.ws_bytes || (pl.num_splits > 1 && !ws))
    return fail(ARGUS_E_WORKSPACE, "decode: workspace %zu bytes < %zu needed", ws_bytes, pl.ws_bytes);
  if (reinterpret_cast<uintptr_t>(ws) & 15) return fail(ARGUS_E_INVALID, "decode: workspace not 16-byte aligned");
  return ARGUS_OK;
}

extern "C" argus_status argus_paged_decode_attn(const argus_decode_args* a, void* ws,
                                                size_t ws_bytes, void* stream) {
  Plan pl;
  argus_status st = plan(a, &pl);
  if (st != ARGUS_OK) return st;
  if (a->batch == 0) return ARGUS_OK;
  if ((st = check_io(a)) != ARGUS_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != ARGUS_OK) return st;
  return run(a, pl, ws, stream);
}

extern "C" argus_status argus_test_decode_stall(const argus_decode_args* a, void* ws, size_t ws_bytes,
                                                uint32_t wait_limit_us, int32_t stall_stage,
                                                void* stream) {
  if (wait_limit_us < 1 || wait_limit_us > 2000000u)
    return fail(ARGUS_E_INVALID, "decode stall test: wait_limit_us %u outside [1, 2000000]", wait_limit_us);
  if (stall_stage < 0) return fail(ARGUS_E_INVALID, "decode stall test: stall_stage must be >= 0");
  if (!a->status) return fail(ARGUS_E_INVALID, "decode stall test: status is required");
  Plan pl;
  argus_status st = plan(a, &pl);
  if (st != ARGUS_OK) return st;
  if (a->batch == 0) return ARGUS_OK;
  if ((st = check_io(a)) != ARGUS_OK) return st;
  if ((st = check_ws(pl, ws, ws_bytes)) != ARGUS_OK) return st;
  return run(a, pl, ws, stream, 1000ull * wait_limit_us, stall_stage);
}

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot hand the library any device memory: runtimes whose
// memory planner has already given out the device memory before decoding
// starts, and host code that must not call cudaMalloc on the decode path
// (cudaMalloc can synchronise the device, and a planner-owned heap has no
// room to spare).  For them the split-combine scratch lives in a fixed
// file-scope device array of ARGUS_NOALLOC_SCRATCH_BYTES bytes, which every
// GPU that loads this library keeps until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[ARGUS_NOALLOC_SCRATCH_BYTES];

namespace argus {
namespace decode {

// Device address of g_noalloc_scratch, resolved with the device current once
// per device and context (the host-side name is only a stand-in for the
// symbol; a context created again after cudaDeviceReset gets a new address).
static argus_status noalloc_scratch(void** out) {
  static void* addr[64] = {};
  static PerContext resolved;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fail(ARGUS_E_LAUNCH, "decode (no-alloc): no current device");
  argus_status st = resolved.ensure([](int d) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      addr[d] = nullptr;
      return fail(ARGUS_E_LAUNCH, "decode (no-alloc): cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    }
    addr[d] = ptr;
    return ARGUS_OK;
  });
  if (st != ARGUS_OK) return st;
  *out = addr[dev];
  return ARGUS_OK;
}

}  // namespace decode
}  // namespace argus

extern "C" argus_status argus_paged_decode_attn_noalloc(const argus_decode_args* a, void* stream) {
  Plan pl;
  argus_status st = plan(a, &pl);
  if (st != ARGUS_OK) return st;
  if (a->batch == 0) return ARGUS_OK;
  if ((st = check_io(a)) != ARGUS_OK) return st;
  if (pl.ws_bytes > (size_t)ARGUS_NOALLOC_SCRATCH_BYTES)
    return fail(ARGUS_E_WORKSPACE,
                "decode (no-alloc): these arguments need %zu bytes of scratch, more than the fixed %zu; "
                "lower num_splits or use argus_paged_decode_attn with a workspace",
                pl.ws_bytes, (size_t)ARGUS_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != ARGUS_OK) return st;
  // the array keeps whatever the previous call left; nothing in it has to
  // start at zero (every partial is written before it is read)
  return run(a, pl, scratch, stream);
}
