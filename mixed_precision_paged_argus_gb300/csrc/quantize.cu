// argus_quantize_pages: demote 16-bit KV pages into a codec tier, bit-exactly.
//
// "ARGUS: Heterogeneous KV-cache memory management" (summary): older pages are
// demoted from FP16 through FP8, INT8 and INT4.  "feat(kvcache): host-RAM KV
// tier for sparse-attention models", update 20f3b23: the pool stores e4m3 codes
// plus fp32 scales and is the source of truth.  Per (page, K|V, KV head) unit:
//   FP8   scale = amax / 448, code = e4m3_rne_satfinite(x / scale)
//   INT8  scale = amax / 127, code = clamp(rint(x / scale), -127, 127)
//   INT4  per token and 32-element group: z = fp16_sat(min),
//         s = fp16_sat((max - z) / 15), code = clamp(rint((x - z) / s), 0, 15)
// every operation IEEE fp32 with round-to-nearest-even.  The quotients are
// formed with a reciprocal product that provably selects the same code as the
// IEEE division, falling back to the division near rounding boundaries.  The optional compressed
// key is the bf16 mean over valid tokens of the stored (dequantised) keys.
//
// GB300 design: the pass is a pure HBM stream.  Units of at most 2048 elements
// are owned by one warp and held in registers (one read, one write); larger
// units are owned by a 256-thread CTA that reads the unit twice (max pass,
// then encode), the second read served from L2.  Loads and stores are 16-byte
// per lane and contiguous across the group.
#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace argus {
namespace quant {

struct QParams {
  int Hkv, P, n_pages;
  const uint16_t* src;
  long long n_src;
  const int32_t* src_slots;
  const int32_t* dst_slots;
  const int32_t* valid_tokens;
  uint8_t* dst_codes;
  uint8_t* dst_meta;
  long long n_dst;
  uint16_t* ckey;
  uint32_t* status;
};

constexpr int kCtaThreads = 256;
constexpr int kRegVecs = 8;  // 16-byte vectors per lane kept in registers (small units)

template <bool SBF16>
__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t bits = (w[e / 2] >> (16 * (e & 1))) & 0xFFFFu;
    f[e] = SBF16 ? __uint_as_float(bits << 16) : __half2float(__ushort_as_half((unsigned short)bits));
  }
}

// |x| maxima and minima on the packed 16-bit sources: non-negative fp16 and
// bf16 values order like their bit patterns, so a packed unsigned max / min of
// the sign-cleared halves finds the largest / smallest magnitude exactly.
template <bool SBF16>
__device__ __forceinline__ float mag_to_float(uint32_t bits16) {
  return SBF16 ? __uint_as_float(bits16 << 16) : __half2float(__ushort_as_half((unsigned short)bits16));
}

__device__ __forceinline__ float fp16_sat(float x) {
  return __half2float(__float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f)));
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t h = e4m3x2_to_f16x2(code & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Reduce over the `group` threads that own one unit (32 = warp, 256 = CTA).
template <int GROUP, bool MAX>
__device__ __forceinline__ float group_reduce(float v, float* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? fmaxf(v, w) : v + w;
  }
  if (GROUP == 32) return v;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  v = sh[0];
#pragma unroll
  for (int w = 1; w < GROUP / 32; ++w) v = MAX ? fmaxf(v, sh[w]) : v + sh[w];
  return v;
}

// Quotients for the encoders.  The codes are defined on RN(x / s) (IEEE fp32
// division).  x * RN(1/s) is within 1.5 ulp of RN(x / s), so it selects the
// same code unless it lies within a few ulps of a rounding boundary of the
// target format.  The encoders form all eight products of a vector, and only
// when one of them is that close (or, for e4m3, in the subnormal range) redo
// the vector with IEEE divisions, on an explicit branch so that the common
// path never evaluates a division.  The codes are therefore identical to
// dividing every element.
//  e4m3 (normal range): boundaries are the midpoints between neighbouring
//  codes, i.e. fp32 mantissas whose 20 bits below the 3 kept bits equal
//  0x80000; a product within 8 of them in those bits, or below 0.0157 in
//  magnitude (e4m3 subnormals start below 2^-6), takes the division.

//  integer codes: boundaries are the half-integers.  For |y| <= 128 the
//  product differs from x / s by at most 128 * 2^-23 = 2^-16 and RN(x / s)
//  from x / s by at most 2^-18, so a product farther than kIntGuard = 2^-14
//  from a half-integer rounds like the quotient.  Rounding to an
//  integer uses the fp32 adder: for |y| < 2^22, y + 1.5 * 2^23 rounds y to the
//  nearest integer (ties to even) and leaves it in the low mantissa bits, so
//  neither a round nor a float-to-int conversion instruction is needed.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kIntGuard = 0x1p-14f;
__device__ __forceinline__ bool rint_unsure(float y, float t) {  // t = y + kRoundMagic
  return fabsf(y - (t - kRoundMagic)) > 0.5f - kIntGuard;
}

// The rare exact path: eight IEEE quotients, kept out of line so that the
// unrolled encoders stay small in the instruction cache.
struct F8 {
  float v[8];
};
__device__ __noinline__ F8 div8(F8 x, float s) {
  F8 q;
#pragma unroll
  for (int e = 0; e < 8; ++e) q.v[e] = x.v[e] / s;
  return q;
}

//  INT4 / INT2 scale: fp16_sat(RN(a / TOP)), TOP = 15 or 3.  a * RN(1/TOP) is
//  within 3 ulp of RN(a/TOP); the fp16 rounding can only differ within a few
//  ulps of an fp16 midpoint (fp32 mantissa bits below the fp16 ones equal to
//  0x1000) or in fp16's subnormal range, where the division itself is taken.
template <int TOP>
__device__ __forceinline__ float scale_div(float a) {
  float y = a * (1.f / (float)TOP);
  const uint32_t low = __float_as_uint(y) & 0x1FFFu;
  if (((low - 0x1000u + 8u) <= 16u) || fabsf(y) < 0x1p-14f) y = a / (float)TOP;
  return fp16_sat(y);
}

// Encode 8 values of one 16-byte source vector and store them; with DEQ the
// stored values are also decoded into deq (for the compressed key).  rscale is
// RN(1 / scale) (FP8, INT8).
template <int CODEC, bool SBF16, bool DEQ>
__device__ __forceinline__ void encode_store(const float (&f)[8], const uint4& raw, float scale, float rscale,
                                             uint8_t* dcodes, size_t vec, bool valid, float (&deq)[8],
                                             uint8_t* dmeta_row, int lane_in_group) {
  if (CODEC == ARGUS_FP16 || CODEC == ARGUS_BF16) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(dcodes)[vec] = valid ? raw : z;
    if (DEQ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) deq[e] = valid ? f[e] : 0.f;
    }
  } else if (CODEC == ARGUS_FP8_E4M3) {
    uint32_t w[2] = {0u, 0u};
    if (valid && scale > 0.f) {
      // the e4m3 boundary test as running minima: of the distance
      // (low mantissa bits - midpoint + 8, unsigned) and of |y|
      float y[8];
      uint32_t dmin = 0xFFFFFFFFu;
#pragma unroll
      for (int e = 0; e < 8; e += 2) f2_mul(y[e], y[e + 1], f[e], f[e + 1], rscale, rscale);
#pragma unroll
      for (int e = 0; e < 8; ++e) dmin = min(dmin, (__float_as_uint(y[e]) & 0xFFFFFu) - 0x80000u + 8u);
      // the smallest |y| is the product of the smallest |x| (the product is
      // monotone in |x|), found on the packed source
      const uint32_t mn2 = __vminu2(__vminu2(raw.x & 0x7FFF7FFFu, raw.y & 0x7FFF7FFFu),
                                    __vminu2(raw.z & 0x7FFF7FFFu, raw.w & 0x7FFF7FFFu));
      const float amin = mag_to_float<SBF16>(min(mn2 & 0xFFFFu, mn2 >> 16)) * rscale;
      if (dmin <= 16u || amin < 0.0157f) {   // near a midpoint, or e4m3 subnormal range
        F8 x;
#pragma unroll
        for (int e = 0; e < 8; ++e) x.v[e] = f[e];
        const F8 q = div8(x, scale);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = q.v[e];
      }
      w[0] = f32x2_to_e4m3x2(y[0], y[1]) | (f32x2_to_e4m3x2(y[2], y[3]) << 16);
      w[1] = f32x2_to_e4m3x2(y[4], y[5]) | (f32x2_to_e4m3x2(y[6], y[7]) << 16);
    }
    if (DEQ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) deq[e] = e4m3_value(w[e / 4] >> (8 * (e & 3))) * scale;
    }
    reinterpret_cast<uint2*>(dcodes)[vec] = make_uint2(w[0], w[1]);
  } else if (CODEC == ARGUS_INT8) {
    uint32_t w[2] = {0u, 0u};
    if (valid && scale > 0.f) {
      // |x * RN(1/s)| <= 127 (1 + 2^-22) while s is a normal number, so the
      // clamp is needed only for the tiny scales of subnormal units; clamping
      // before rounding equals clamping the rounded value (integer bounds)
      uint32_t t[8];
      float dev = 0.f;   // largest distance of a product from its rounded value
      auto round8 = [&](auto clamp_tag) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          float y0, y1, t0, t1, q0, q1, e0, e1;
          f2_mul(y0, y1, f[e], f[e + 1], rscale, rscale);
          if (decltype(clamp_tag)::value) {
            y0 = fminf(fmaxf(y0, -127.f), 127.f);
            y1 = fminf(fmaxf(y1, -127.f), 127.f);
          }
          f2_add(t0, t1, y0, y1, kRoundMagic, kRoundMagic);
          f2_sub(q0, q1, t0, t1, kRoundMagic, kRoundMagic);
          f2_sub(e0, e1, y0, y1, q0, q1);
          dev = fmaxf(dev, fmaxf(fabsf(e0), fabsf(e1)));
          t[e] = __float_as_uint(t0);
          t[e + 1] = __float_as_uint(t1);
        }
      };
      if (scale < 0x1p-100f) round8(std::true_type{});   // the branch stays outside the loop
      else round8(std::false_type{});
      if (dev > 0.5f - kIntGuard) {
        F8 x;
#pragma unroll
        for (int e = 0; e < 8; ++e) x.v[e] = f[e];
        const F8 q = div8(x, scale);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = __float_as_uint(fminf(fmaxf(q.v[e], -127.f), 127.f) + kRoundMagic);
      }
      // the low byte of the mantissa is the code in two's complement
      w[0] = prmt(prmt(t[0], t[1], 0x0040), prmt(t[2], t[3], 0x0040), 0x5410);
      w[1] = prmt(prmt(t[4], t[5], 0x0040), prmt(t[6], t[7], 0x0040), 0x5410);
    }
    if (DEQ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) deq[e] = (float)(int8_t)((w[e / 4] >> (8 * (e & 3))) & 0xFF) * scale;
    }
    reinterpret_cast<uint2*>(dcodes)[vec] = make_uint2(w[0], w[1]);
  } else {  // INT4 / INT2 / INT1: the 4 threads of a 32-element group cooperate
    constexpr int BITS = (CODEC == ARGUS_INT4_G32) ? 4 : (CODEC == ARGUS_INT2_G32 ? 2 : 1);
    constexpr int TOP = (1 << BITS) - 1;
    constexpr uint32_t MASK = (uint32_t)TOP;
    float lo = f[0], hi = f[0];
#pragma unroll
    for (int e = 1; e < 8; ++e) {
      lo = fminf(lo, f[e]);
      hi = fmaxf(hi, f[e]);
    }
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 1));
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, 2));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, 2));
    const float z = fp16_sat(lo);
    const float s = scale_div<TOP>(hi - z);
    uint32_t w = 0u;
    if (valid && s > 0.f) {
      const float r = __frcp_rn(s);
      float d[8];
      uint32_t t[8];
      bool unsure = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        d[e] = f[e] - z;
        const float y = fminf(fmaxf(d[e] * r, 0.f), (float)TOP);
        const float tf = y + kRoundMagic;
        unsure |= rint_unsure(y, tf);
        t[e] = __float_as_uint(tf);
      }
      if (unsure) {
        F8 x;
#pragma unroll
        for (int e = 0; e < 8; ++e) x.v[e] = d[e];
        const F8 q = div8(x, s);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = __float_as_uint(fminf(fmaxf(q.v[e], 0.f), (float)TOP) + kRoundMagic);
      }
      // code e of the 8 at bits BITS * e: INT4 even elements in the low
      // nibbles, INT2 element 4k + j at bits 2j of byte k, INT1 element e at bit e
#pragma unroll
      for (int e = 0; e < 8; ++e) w |= (t[e] & MASK) << (BITS * e);
    }
    const float zz = valid ? z : 0.f, ss = valid ? s : 0.f;
    if (DEQ) {
#pragma unroll
      for (int e = 0; e < 8; ++e) deq[e] = fmaf((float)((w >> (BITS * e)) & MASK), ss, zz);
    }
    if (BITS == 4) reinterpret_cast<uint32_t*>(dcodes)[vec] = w;
    else if (BITS == 2) reinterpret_cast<uint16_t*>(dcodes)[vec] = (uint16_t)w;
    else dcodes[vec] = (uint8_t)w;
    if ((lane_in_group & 3) == 0) {
      const __half2 sz = __halves2half2(__float2half_rn(ss), __float2half_rn(zz));
      *reinterpret_cast<__half2*>(dmeta_row) = sz;
    }
  }
}

template <int D, bool SBF16, int CODEC, int GROUP>
__global__ void __launch_bounds__(kCtaThreads) quantize_kernel(const QParams p) {
  constexpr int VPR = D / 8;  // 16-byte vectors per token row
  __shared__ float sh_red[kCtaThreads / 32];
  __shared__ float sh_ck[kCtaThreads / 32][8 * VPR];
  const int lane = threadIdx.x & 31;
  const int g = (GROUP == 32) ? lane : threadIdx.x;
  const long long gid = (GROUP == 32) ? (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5)
                                      : (long long)blockIdx.x;
  const long long ngroups = (GROUP == 32) ? (long long)gridDim.x * (blockDim.x / 32) : gridDim.x;
  const int Hkv = p.Hkv, P = p.P;
  const long long n_units = (long long)p.n_pages * 2 * Hkv;
  const int nvec = P * VPR;  // vectors per unit

  for (long long u = gid; u < n_units; u += ngroups) {
    const int i = (int)(u / (2 * Hkv));
    const int rem = (int)(u - (long long)i * 2 * Hkv);
    const int kv = rem / Hkv, h = rem - kv * Hkv;
    const long long ss = p.src_slots[i], ds = p.dst_slots[i];
    if (ss < 0 || ss >= p.n_src || ds < 0 || ds >= p.n_dst) {
      if (g == 0 && kv == 0 && h == 0 && p.status) atomicAdd(p.status, 1u);
      continue;
    }
    int valid = p.valid_tokens ? p.valid_tokens[i] : P;
    valid = max(0, min(P, valid));
    const int nvalid_vec = valid * VPR;
    const uint4* src = reinterpret_cast<const uint4*>(p.src + ((ss * 2 + kv) * Hkv + h) * (size_t)P * D);
    const size_t unit_dst = ((size_t)ds * 2 + kv) * Hkv + h;
    uint8_t* dcodes;
    if (CODEC == ARGUS_FP16 || CODEC == ARGUS_BF16) dcodes = p.dst_codes + unit_dst * (size_t)P * D * 2;
    else if (CODEC == ARGUS_INT4_G32) dcodes = p.dst_codes + unit_dst * (size_t)P * (D / 2);
    else if (CODEC == ARGUS_INT2_G32) dcodes = p.dst_codes + unit_dst * (size_t)P * (D / 4);
    else if (CODEC == ARGUS_INT1_G32) dcodes = p.dst_codes + unit_dst * (size_t)P * (D / 8);
    else dcodes = p.dst_codes + unit_dst * (size_t)P * D;

    const bool regs = (GROUP == 32) && (nvec <= 32 * kRegVecs);
    uint4 held[kRegVecs];
    float scale = 0.f;
    if (CODEC == ARGUS_FP8_E4M3 || CODEC == ARGUS_INT8) {
      float amax = 0.f;
      if (regs) {
#pragma unroll
        for (int k = 0; k < kRegVecs; ++k) {
          const int v = g + 32 * k;
          if (v < nvec) {
            held[k] = src[v];
            if (v < nvalid_vec) {
              float f[8];
              unpack8<SBF16>(held[k], f);
#pragma unroll
              for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
            }
          }
        }
      } else {
        for (int v = g; v < nvalid_vec; v += GROUP) {
          float f[8];
          unpack8<SBF16>(src[v], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
        }
      }
      amax = group_reduce<GROUP, true>(amax, sh_red);
      scale = amax > 0.f ? amax / (CODEC == ARGUS_FP8_E4M3 ? 448.f : 127.f) : 0.f;
      if (g == 0) reinterpret_cast<float*>(p.dst_meta)[unit_dst] = scale;
    }
    const float rscale = scale > 0.f ? 1.f / scale : 0.f;

    float ck[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto do_vec = [&](int v, const uint4& raw) {
      float f[8];
      unpack8<SBF16>(raw, f);
      const bool valid_v = v < nvalid_vec;
      float deq[8];
      uint8_t* meta_row = nullptr;
      if (CODEC == ARGUS_INT4_G32 || CODEC == ARGUS_INT2_G32 || CODEC == ARGUS_INT1_G32) {
        const int row = v / VPR, grp = (v % VPR) / 4;
        meta_row = p.dst_meta + ((unit_dst * P + row) * (D / 32) + grp) * 4;
      }
      encode_store<CODEC, SBF16, true>(f, raw, scale, rscale, dcodes, (size_t)v, valid_v, deq, meta_row, g);
      if (valid_v) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ck[e] += deq[e];
      }
    };
    if (regs) {
      if (!(CODEC == ARGUS_FP8_E4M3 || CODEC == ARGUS_INT8)) {
#pragma unroll
        for (int k = 0; k < kRegVecs; ++k) {
          const int v = g + 32 * k;
          if (v < nvec) held[k] = src[v];
        }
      }
#pragma unroll
      for (int k = 0; k < kRegVecs; ++k) {
        const int v = g + 32 * k;
        if (v < nvec) do_vec(v, held[k]);
      }
    } else {
      for (int v = g; v < nvec; v += GROUP) do_vec(v, src[v]);
    }

    if (p.ckey && kv == 0) {
      // threads with equal g % VPR hold the same 8 dims
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float x = ck[e];
#pragma unroll
        for (int o = VPR; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        ck[e] = x;
      }
      if (GROUP != 32) {
        const int warp = threadIdx.x >> 5;
        __syncthreads();
        if (lane < VPR) {
#pragma unroll
          for (int e = 0; e < 8; ++e) sh_ck[warp][lane * 8 + e] = ck[e];
        }
        __syncthreads();
        if (threadIdx.x < VPR) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float x = 0.f;
            for (int w = 0; w < GROUP / 32; ++w) x += sh_ck[w][threadIdx.x * 8 + e];
            ck[e] = x;
          }
        }
      }
      if (g < VPR) {
        const float n_f = (float)max(valid, 1);
        uint32_t outw[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float a0 = valid ? ck[e] / n_f : 0.f;
          const float a1 = valid ? ck[e + 1] / n_f : 0.f;
          outw[e / 2] = pack_bf16x2(a0, a1);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.ckey + ((size_t)i * Hkv + h) * D);
        dst[g] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
      }
    }
    if (GROUP != 32) __syncthreads();
  }
}

// INT4 / INT2 / INT1 with one lane per 32-element group (the group's four
// 16-byte source vectors in x0..x3): the min / max reduction and the scale
// arithmetic are lane-local and done once per group, and the 32 codes leave as
// one store (16 bytes of INT4 in w[0..3], 8 bytes of INT2 in w[0..1], 4 bytes
// of INT1 in w[0]).  Same arithmetic, hence the same codes, as encode_store's
// affine path.
template <bool SBF16, int BITS>
__device__ __forceinline__ void encode_affine_group(const uint4 (&x)[4], bool valid, uint32_t (&wout)[4],
                                                    uint32_t& meta) {
  constexpr int TOP = (1 << BITS) - 1;
  uint32_t mn, mx;
  {
    const uint32_t* wv = reinterpret_cast<const uint32_t*>(&x[0]);
    if (SBF16) {
      __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&wv[0]), b = a;
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&wv[i]);
        a = __hmin2(a, c);
        b = __hmax2(b, c);
      }
      mn = *reinterpret_cast<uint32_t*>(&a);
      mx = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 a = *reinterpret_cast<const __half2*>(&wv[0]), b = a;
#pragma unroll
      for (int i = 1; i < 16; ++i) {
        const __half2 c = *reinterpret_cast<const __half2*>(&wv[i]);
        a = __hmin2(a, c);
        b = __hmax2(b, c);
      }
      mn = *reinterpret_cast<uint32_t*>(&a);
      mx = *reinterpret_cast<uint32_t*>(&b);
    }
  }
  auto to_f = [](uint32_t bits16) -> float {
    return SBF16 ? __uint_as_float(bits16 << 16) : __half2float(__ushort_as_half((unsigned short)bits16));
  };
  const float lo = fminf(to_f(mn & 0xFFFFu), to_f(mn >> 16));
  const float hi = fmaxf(to_f(mx & 0xFFFFu), to_f(mx >> 16));
  const float z = fp16_sat(lo);
  const float s = scale_div<TOP>(hi - z);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (valid && s > 0.f) {
    const float r = __frcp_rn(s);
    // the products are monotone in x: when those of the group's min and max
    // round into 0..TOP, no product needs the clamp
    const bool clamp = !((lo - z) * r > -0.49f && (hi - z) * r < (float)TOP + 0.49f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float f[8], d[8];
      uint32_t t[8];
      unpack8<SBF16>(x[m], f);
      float dev = 0.f;  // largest distance of a product from its rounded value
      // element pairs in packed f32x2 instructions (the same IEEE operations)
      auto round8 = [&](auto clamp_tag) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          f2_sub(d[e], d[e + 1], f[e], f[e + 1], z, z);
          float y0, y1, t0, t1, q0, q1, e0, e1;
          f2_mul(y0, y1, d[e], d[e + 1], r, r);
          if (decltype(clamp_tag)::value) {
            y0 = fminf(fmaxf(y0, 0.f), (float)TOP);
            y1 = fminf(fmaxf(y1, 0.f), (float)TOP);
          }
          f2_add(t0, t1, y0, y1, kRoundMagic, kRoundMagic);
          f2_sub(q0, q1, t0, t1, kRoundMagic, kRoundMagic);
          f2_sub(e0, e1, y0, y1, q0, q1);
          dev = fmaxf(dev, fmaxf(fabsf(e0), fabsf(e1)));
          t[e] = __float_as_uint(t0);
          t[e + 1] = __float_as_uint(t1);
        }
      };
      if (clamp) round8(std::true_type{});
      else round8(std::false_type{});
      if (dev > 0.5f - kIntGuard) {
        F8 x;
#pragma unroll
        for (int e = 0; e < 8; ++e) x.v[e] = d[e];
        const F8 q = div8(x, s);
#pragma unroll
        for (int e = 0; e < 8; ++e) t[e] = __float_as_uint(fminf(fmaxf(q.v[e], 0.f), (float)TOP) + kRoundMagic);
      }
      if (BITS == 4) {
        // low bytes of t are the codes 0..15: even elements in the low nibbles
        const uint32_t ev = prmt(prmt(t[0], t[2], 0x0040), prmt(t[4], t[6], 0x0040), 0x5410);
        const uint32_t od = prmt(prmt(t[1], t[3], 0x0040), prmt(t[5], t[7], 0x0040), 0x5410);
        w[m] = ev + (od << 4);
      } else if (BITS == 2) {
        // codes 0..3: byte 0 takes elements 0..3, byte 1 elements 4..7, element
        // j of a byte at bits 2j; xj holds elements j and 4 + j in bytes 0, 1
        const uint32_t x0 = prmt(t[0], t[4], 0x0040), x1 = prmt(t[1], t[5], 0x0040);
        const uint32_t x2 = prmt(t[2], t[6], 0x0040), x3 = prmt(t[3], t[7], 0x0040);
        const uint32_t w16 = (x0 | (x1 << 2) | (x2 << 4) | (x3 << 6)) & 0xFFFFu;
        w[m >> 1] |= w16 << (16 * (m & 1));
      } else {
        // codes 0..1: vector m's eight elements fill byte m, element e at bit e
        uint32_t b = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) b |= (t[e] & 1u) << e;
        w[0] |= b << (8 * m);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) wout[k] = w[k];
  const __half2 sz = __halves2half2(__float2half_rn(valid ? s : 0.f), __float2half_rn(valid ? z : 0.f));
  meta = *reinterpret_cast<const uint32_t*>(&sz);
}

// Units of at most 2048 elements: one warp per unit, held in registers,
// software-pipelined so that the next unit's loads are in flight while the
// current one is reduced, encoded and stored.
// CK: compressed keys requested (the kernel is instantiated for both, so that
// the common case carries no decode-and-sum code)
template <int D, bool SBF16, int CODEC, bool CK>
__global__ void __launch_bounds__(kCtaThreads) quantize_small_kernel(const QParams p) {
  constexpr int VPR = D / 8;
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const long long nw = (long long)gridDim.x * (blockDim.x / 32);
  const int Hkv = p.Hkv, P = p.P;
  const long long n_units = (long long)p.n_pages * 2 * Hkv;
  const int nvec = P * VPR;
  constexpr bool want_ck = CK;

  struct Unit {
    const uint4* src;
    size_t dst;
    int page, kv, h, valid;
    bool ok;
  };
  auto describe = [&](long long u) {
    Unit d;
    d.page = (int)(u / (2 * Hkv));
    const int rem = (int)(u - (long long)d.page * 2 * Hkv);
    d.kv = rem / Hkv;
    d.h = rem - d.kv * Hkv;
    const long long ss = p.src_slots[d.page], ds = p.dst_slots[d.page];
    d.ok = !(ss < 0 || ss >= p.n_src || ds < 0 || ds >= p.n_dst);
    int valid = p.valid_tokens ? p.valid_tokens[d.page] : P;
    d.valid = max(0, min(P, valid));
    d.src = reinterpret_cast<const uint4*>(p.src + ((ss * 2 + d.kv) * Hkv + d.h) * (size_t)P * D);
    d.dst = ((size_t)ds * 2 + d.kv) * Hkv + d.h;
    return d;
  };
  constexpr bool want_ck_any = CK;
  // INT4 units without a compressed key use one lane per 32-element group:
  // slot 4j + m holds vector m of group lane + 32j
  auto group_layout = [&](const Unit& d) {
    return (CODEC == ARGUS_INT4_G32 || CODEC == ARGUS_INT2_G32 || CODEC == ARGUS_INT1_G32) &&
           !(want_ck_any && d.kv == 0);
  };
  auto load = [&](const Unit& d, uint4 (&buf)[kRegVecs]) {
    const bool gl = group_layout(d);
#pragma unroll
    for (int k = 0; k < kRegVecs; ++k) {
      const int v = gl ? 4 * (lane + 32 * (k >> 2)) + (k & 3) : lane + 32 * k;
      if (d.ok && v < nvec) buf[k] = __ldcs(d.src + v);   // streamed once: evict first
    }
  };

  long long u = wid;
  if (u >= n_units) return;
  uint4 cur[kRegVecs], nxt[kRegVecs];
  Unit cu = describe(u);
  load(cu, cur);
  while (u < n_units) {
    const long long un = u + nw;
    Unit nu = cu;
    if (un < n_units) {
      nu = describe(un);
      load(nu, nxt);
    }
    if (!cu.ok) {
      if (lane == 0 && cu.kv == 0 && cu.h == 0 && p.status) atomicAdd(p.status, 1u);
    } else if (group_layout(cu)) {
      constexpr int GPR = D / 32;  // groups per token row
      constexpr int BITS = (CODEC == ARGUS_INT4_G32) ? 4 : (CODEC == ARGUS_INT2_G32 ? 2 : 1);
      uint8_t* gcodes = p.dst_codes + cu.dst * (size_t)P * (D * BITS / 8);
      uint32_t* gmeta = reinterpret_cast<uint32_t*>(p.dst_meta) + cu.dst * (size_t)P * GPR;
#pragma unroll
      for (int j = 0; j < kRegVecs / 4; ++j) {
        const int idx = lane + 32 * j;
        if (4 * idx < nvec) {
          const uint4 xg[4] = {cur[4 * j], cur[4 * j + 1], cur[4 * j + 2], cur[4 * j + 3]};
          uint32_t c[4];
          uint32_t m;
          encode_affine_group<SBF16, BITS>(xg, idx / GPR < cu.valid, c, m);
          if (BITS == 4) reinterpret_cast<uint4*>(gcodes)[idx] = make_uint4(c[0], c[1], c[2], c[3]);
          else if (BITS == 2) reinterpret_cast<uint2*>(gcodes)[idx] = make_uint2(c[0], c[1]);
          else reinterpret_cast<uint32_t*>(gcodes)[idx] = c[0];
          gmeta[idx] = m;
        }
      }
    } else {
      const int nvalid_vec = cu.valid * VPR;
      uint8_t* dcodes;
      if (CODEC == ARGUS_FP16 || CODEC == ARGUS_BF16) dcodes = p.dst_codes + cu.dst * (size_t)P * D * 2;
      else if (CODEC == ARGUS_INT4_G32) dcodes = p.dst_codes + cu.dst * (size_t)P * (D / 2);
      else if (CODEC == ARGUS_INT2_G32) dcodes = p.dst_codes + cu.dst * (size_t)P * (D / 4);
      else if (CODEC == ARGUS_INT1_G32) dcodes = p.dst_codes + cu.dst * (size_t)P * (D / 8);
      else dcodes = p.dst_codes + cu.dst * (size_t)P * D;
      float scale = 0.f;
      if (CODEC == ARGUS_FP8_E4M3 || CODEC == ARGUS_INT8) {
        uint32_t mx2 = 0u;   // per 16-bit half: the largest sign-cleared code
#pragma unroll
        for (int k = 0; k < kRegVecs; ++k) {
          const int v = lane + 32 * k;
          if (v < nvalid_vec) {
            const uint4 x = cur[k];
            mx2 = __vmaxu2(mx2, __vmaxu2(__vmaxu2(x.x & 0x7FFF7FFFu, x.y & 0x7FFF7FFFu),
                                         __vmaxu2(x.z & 0x7FFF7FFFu, x.w & 0x7FFF7FFFu)));
          }
        }
        float amax = mag_to_float<SBF16>(max(mx2 & 0xFFFFu, mx2 >> 16));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        scale = amax > 0.f ? amax / (CODEC == ARGUS_FP8_E4M3 ? 448.f : 127.f) : 0.f;
        if (lane == 0) reinterpret_cast<float*>(p.dst_meta)[cu.dst] = scale;
      }
      const float rscale = scale > 0.f ? 1.f / scale : 0.f;
      float ck[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // decoding the stored values is needed only for a compressed key
      auto encode_unit = [&](auto deq_tag) {
        constexpr bool DEQ = decltype(deq_tag)::value;
#pragma unroll
        for (int k = 0; k < kRegVecs; ++k) {
          const int v = lane + 32 * k;
          if (v < nvec) {
            float f[8], deq[8];
            unpack8<SBF16>(cur[k], f);
            uint8_t* meta_row = nullptr;
            if (CODEC == ARGUS_INT4_G32 || CODEC == ARGUS_INT2_G32 || CODEC == ARGUS_INT1_G32) {
              const int row = v / VPR, grp = (v % VPR) / 4;
              meta_row = p.dst_meta + ((cu.dst * P + row) * (D / 32) + grp) * 4;
            }
            const bool valid_v = v < nvalid_vec;
            encode_store<CODEC, SBF16, DEQ>(f, cur[k], scale, rscale, dcodes, (size_t)v, valid_v, deq, meta_row,
                                            lane);
            if (DEQ && valid_v) {
#pragma unroll
              for (int e = 0; e < 8; ++e) ck[e] += deq[e];
            }
          }
        }
      };
      const bool ck_unit = want_ck && cu.kv == 0;
      if (ck_unit) encode_unit(std::true_type{});
      else encode_unit(std::false_type{});
      if (ck_unit) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float x = ck[e];
#pragma unroll
          for (int o = VPR; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
          ck[e] = x;
        }
        if (lane < VPR) {
          const float n_f = (float)max(cu.valid, 1);
          uint32_t outw[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float a0 = cu.valid ? ck[e] / n_f : 0.f;
            const float a1 = cu.valid ? ck[e + 1] / n_f : 0.f;
            outw[e / 2] = pack_bf16x2(a0, a1);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.ckey + ((size_t)cu.page * Hkv + cu.h) * D);
          dst[lane] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        }
      }
    }
    u = un;
    cu = nu;
#pragma unroll
    for (int k = 0; k < kRegVecs; ++k) cur[k] = nxt[k];
  }
}

template <int D, bool SBF16, int CODEC>
static argus_status launch3(const QParams& p, cudaStream_t s) {
  const long long units = (long long)p.n_pages * 2 * p.Hkv;
  const int sms = device_sm_count();
  const bool small = (long long)p.P * D <= 32 * kRegVecs * 8;
  if (small) {
    const long long blocks_needed = (units + (kCtaThreads / 32) - 1) / (kCtaThreads / 32);
    // one wave: two CTAs per SM are resident at this kernel's register count
    const int blocks = (int)std::max<long long>(1, std::min<long long>(blocks_needed, (long long)sms * 2));
    if (p.ckey) quantize_small_kernel<D, SBF16, CODEC, true><<<blocks, kCtaThreads, 0, s>>>(p);
    else quantize_small_kernel<D, SBF16, CODEC, false><<<blocks, kCtaThreads, 0, s>>>(p);
  } else {
    const int blocks = (int)std::max<long long>(1, std::min<long long>(units, (long long)sms * 8));
    quantize_kernel<D, SBF16, CODEC, kCtaThreads><<<blocks, kCtaThreads, 0, s>>>(p);
  }
  return launch_status("argus_quantize_pages");
}

template <int D, bool SBF16>
static argus_status launch2(int codec, const QParams& p, cudaStream_t s) {
  switch (codec) {
    case ARGUS_FP16: return launch3<D, SBF16, ARGUS_FP16>(p, s);
    case ARGUS_BF16: return launch3<D, SBF16, ARGUS_BF16>(p, s);
    case ARGUS_FP8_E4M3: return launch3<D, SBF16, ARGUS_FP8_E4M3>(p, s);
    case ARGUS_INT8: return launch3<D, SBF16, ARGUS_INT8>(p, s);
    case ARGUS_INT2_G32: return launch3<D, SBF16, ARGUS_INT2_G32>(p, s);
    case ARGUS_INT1_G32: return launch3<D, SBF16, ARGUS_INT1_G32>(p, s);
    default: return launch3<D, SBF16, ARGUS_INT4_G32>(p, s);
  }
}

}  // namespace quant
}  // namespace argus

using namespace argus;
using namespace argus::quant;

extern "C" argus_status argus_quantize_pages(const argus_geom* g, int32_t src_dtype,
                                             const void* src_codes, int64_t n_src_slots,
                                             const int32_t* src_slots, const argus_pool* dst,
                                             const int32_t* dst_slots, int32_t n_pages,
                                             const int32_t* valid_tokens, void* ckey_out,
                                             uint32_t* status, void* stream) {
  if (!g || !dst) return fail(ARGUS_E_INVALID, "quantize: geometry or destination is NULL");
  if (g->n_kv_heads <= 0 || g->head_dim <= 0 || g->page_tokens <= 0)
    return fail(ARGUS_E_INVALID, "quantize: geometry fields must be positive");
  if (g->head_dim != 64 && g->head_dim != 128)
    return fail(ARGUS_E_UNSUPPORTED, "quantize: head_dim %d (supported: 64, 128)", g->head_dim);
  if (src_dtype != ARGUS_FP16 && src_dtype != ARGUS_BF16)
    return fail(ARGUS_E_INVALID, "quantize: src_dtype must be FP16 or BF16");
  if (dst->codec < 0 || dst->codec > ARGUS_INT1_G32) return fail(ARGUS_E_INVALID, "quantize: bad destination codec");
  if ((dst->codec == ARGUS_FP16 || dst->codec == ARGUS_BF16) && dst->codec != src_dtype)
    return fail(ARGUS_E_UNSUPPORTED, "quantize: a 16-bit destination must match the source dtype");
  if (n_pages < 0) return fail(ARGUS_E_INVALID, "quantize: negative n_pages");
  if (n_pages == 0) return ARGUS_OK;
  if (!src_codes || !src_slots || !dst_slots || !dst->codes)
    return fail(ARGUS_E_INVALID, "quantize: NULL source, slot list or destination codes");
  if (dst->codec >= ARGUS_FP8_E4M3 && !dst->meta) return fail(ARGUS_E_INVALID, "quantize: NULL destination meta");
  if ((reinterpret_cast<uintptr_t>(src_codes) | reinterpret_cast<uintptr_t>(dst->codes) |
       reinterpret_cast<uintptr_t>(ckey_out)) & 15)
    return fail(ARGUS_E_INVALID, "quantize: pointers must be 16-byte aligned");
  if (dst->meta && (reinterpret_cast<uintptr_t>(dst->meta) & 3))
    return fail(ARGUS_E_INVALID, "quantize: meta must be 4-byte aligned");
  if ((long long)n_pages * 2 * g->n_kv_heads > (1LL << 31))
    return fail(ARGUS_E_UNSUPPORTED, "quantize: too many units");
  QParams p{};
  p.Hkv = g->n_kv_heads;
  p.P = g->page_tokens;
  p.n_pages = n_pages;
  p.src = static_cast<const uint16_t*>(src_codes);
  p.n_src = n_src_slots;
  p.src_slots = src_slots;
  p.dst_slots = dst_slots;
  p.valid_tokens = valid_tokens;
  // a destination pool in host memory (the host tier) is written in place
  const void* dcodes = nullptr;
  const void* dmeta = nullptr;
  argus_status stp = pool_device_ptrs(*dst, &dcodes, &dmeta);
  if (stp != ARGUS_OK) return stp;
  p.dst_codes = static_cast<uint8_t*>(const_cast<void*>(dcodes));
  p.dst_meta = static_cast<uint8_t*>(const_cast<void*>(dmeta));
  p.n_dst = dst->n_slots;
  p.ckey = static_cast<uint16_t*>(ckey_out);
  p.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = (src_dtype == ARGUS_BF16);
  if (g->head_dim == 64) return bf ? launch2<64, true>(dst->codec, p, s) : launch2<64, false>(dst->codec, p, s);
  return bf ? launch2<128, true>(dst->codec, p, s) : launch2<128, false>(dst->codec, p, s);
}
