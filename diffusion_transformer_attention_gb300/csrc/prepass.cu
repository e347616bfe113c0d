// SAGE quantize prepass: memory-bound kernels that read bf16 Q/K/V once or twice and write
// 1-byte (or exactly-widened 2-byte) codes plus float32 scales.
//
// What they compute follows "VisualGen Quantized Attention", section "SageAttention in the
// TRTLLM backend" (one scale per token block per head for Q and K; V per head per channel in
// FP8 E4M3) and the "TRTLLM Attention" user guide, section "SAGE quantization" (K-smoothing is
// internal). Where the pages are silent the kernels take these readings, which the oracle
// shares and the parity tests check bit for bit:
//   * the K mean is over all Skv tokens: float64 partial sums in a fixed order, divided by Skv
//     in float64, rounded once to float32; smoothed K = float32(K) - mean (float32 subtract);
//   * scale = absmax / QMAX (QMAX 127 or 448) and code = f(x / scale), both IEEE float32
//     divisions (true division, round to nearest); INT8 rounds half to even and clamps to
//     +-127; E4M3 rounds to nearest even and saturates, and a quotient of -0 gives 0x80; an
//     all-zero block has scale 0 and zero codes. The quotients x / scale are computed from the
//     scale's correctly rounded reciprocal with two remainder corrections (quant_math.cuh),
//     which gives the same codes.
//
// Access pattern: a row of one head is 128 bf16 = 256 contiguous bytes. The quantizers read it with
// 16 lanes and 16-byte vector loads (a warp covers two rows per instruction) and write codes with
// 8-byte (or, widened, 16-byte) stores at the same positions; the statistics pass reads it with a
// whole warp and 8-byte loads. Each thread issues several rows' loads before it uses any of them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "ditattn_internal.h"
#include "quant_math.cuh"

namespace ditattn {
namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Programmatic dependent launch. A kernel launched with the programmatic stream serialization
// attribute may start once every CTA of the kernel before it in the stream has started or exited
// and executed launch_dependents; griddepcontrol.wait then returns once that kernel has completed
// and its writes are visible. Under an ordinary launch both are no-ops. The statistics kernels and
// the quantizers call launch_dependents first; a kernel that reads the one before it waits first,
// and a quantizer waits last: the next kernel may fill the SMs a last wave leaves idle, and each
// kernel still completes only after the kernel before it, so an ordinary launch that follows the
// chain waits for all of it.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// x / scale for a scale whose reciprocal rcp was taken when fast (see quant_math.cuh); 0 for a
// zero scale.
__device__ __forceinline__ float quotient(float x, float scale, bool fast, float rcp) {
  if (fast) return div_by_scale(x, scale, rcp);
  return (scale == 0.0f) ? 0.0f : __fdiv_rn(x, scale);
}

// quotient() of a lane's eight values by one block scale, two at a time on the packed pipes. For
// INT8 codes the sign of a zero quotient does not matter (div2_by_scale's ZERO_SIGN is off) and the
// quotients are left in [-127.5, 127.5], where int8_round2 needs them: with the scale amax / 127
// rounded to a normal float32 (every fast scale), |x / scale| <= 127 (1 + 2^-24) and its rounding
// stays below 127.5; a subnormal scale (the IEEE path) can be far smaller than amax / 127, so there
// the quotient is clamped to [-127, 127], which gives the same code as clamping the rounded value.
template <bool INT8_CODES>
__device__ __forceinline__ void quotients8(float* q, float scale, bool fast, float rcp) {
  if (fast) {
    const float2 s2 = make_float2(scale, scale), r2 = make_float2(rcp, rcp);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float2 v = div2_by_scale<!INT8_CODES>(make_float2(q[e], q[e + 1]), s2, r2);
      q[e] = v.x;
      q[e + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      q[e] = (scale == 0.0f) ? 0.0f : __fdiv_rn(q[e], scale);
      if constexpr (INT8_CODES) q[e] = fminf(fmaxf(q[e], -127.0f), 127.0f);
    }
  }
}

// INT8 codes without the conversion unit. Adding 1.5 * 2^23 to a float32 of magnitude <= 2^22
// rounds it to an integer, half to even (the sum's unit in the last place is 1), and leaves that
// integer n in the low mantissa bits: the sum's bits are 0x4B400000 + n. The quotients come from
// quotients8<true>, within [-127.5, 127.5), so n is in [-127, 127] without a clamp. Two values at a
// time: the addition runs on the packed float32 pipes (each lane rounds as the scalar add would).
constexpr float kRoundInt = 12582912.0f;  // 1.5 * 2^23
__device__ __forceinline__ float2 int8_round2(float a, float b) {
  return __fadd2_rn(make_float2(a, b), make_float2(kRoundInt, kRoundInt));
}

// Four INT8 codes, `a` in the low byte (the low byte of the rounded sum is n's two's complement).
__device__ __forceinline__ uint32_t int8_codes4(float a, float b, float c, float d) {
  const float2 ab = int8_round2(a, b), cd = int8_round2(c, d);
  return __byte_perm(__byte_perm(__float_as_uint(ab.x), __float_as_uint(ab.y), 0x0040),
                     __byte_perm(__float_as_uint(cd.x), __float_as_uint(cd.y), 0x0040), 0x5410);
}

// Two INT8 codes held exactly as fp16, `lo` in bits 0-15 (a zero code is +0).
__device__ __forceinline__ uint32_t int8_code_f16x2(float lo, float hi) {
  const float2 n = __fadd2_rn(int8_round2(lo, hi), make_float2(-kRoundInt, -kRoundInt));
  const __half2 h2 = __floats2half2_rn(n.x, n.y);
  return *reinterpret_cast<const uint32_t*>(&h2);
}

// ------------------------------------------------------------------ K mean / V absmax
// Exact float32 sums of K by splitting each value over three levels. For a float32 r with
// |r| <= 2^(k-6) and C = 1.5 * 2^k, r + C lies in [2^k, 2^(k+1)), where the unit in the last place
// is g = 2^(k-23): (r + C) - C is exact (Sterbenz) and equals hi, r rounded to a multiple of g, and
// r - hi (at most g/2 in magnitude, the low-order bits of r) is exact as well. A level's
// accumulator adds 128 such hi values, multiples of g no larger than 2^17 g, so every partial sum
// is a multiple of g of magnitude <= 2^24 g: float32 adds them without rounding. Level k takes the
// remainder of the level before it (at most 2^(k-6) when k drops by 18 per level): with k = 24, 6,
// -12 the levels' grids are 2^1, 2^-17 and 2^-35, and every bf16 value with |x| <= 2^18 whose
// lowest set bit is at least 2^-35 (every such |x| >= 2^-28) is split with remainder 0. A CTA
// that meets anything else (larger values, smaller bits, subnormals, Inf or NaN) sums its tokens
// in float64 instead, in token order. GB300's float64 rate is low, so this keeps the per-element
// work on the packed float32 pipes: four packed operations per level and channel pair.
constexpr int kSplitLevels = 3;
__device__ __forceinline__ constexpr float split_c(int i) {  // C = 1.5 * 2^k for k = 24, 6, -12
  return i == 0 ? 0x1.8p+24f : (i == 1 ? 0x1.8p+6f : 0x1.8p-12f);
}
constexpr uint32_t kSplitMaxAbs = 0x48804880u;  // 2^18 in both bf16 halves
constexpr int kStatsBatch = 8;  // token rows a lane loads before it adds them (loads in flight)

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ __nv_bfloat162 u32_as_bf162(uint32_t u) {
  __nv_bfloat162 r;
  memcpy(&r, &u, sizeof(r));
  return r;
}

__device__ __forceinline__ void bf16x4_to_f32(const uint2& u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xFFFF0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

// Splits a pair of K values (one bf16x2 word) into the levels' accumulators; ORs the bits of the
// final remainders into rem (zero while every value was split exactly, up to the sign of zero).
__device__ __forceinline__ void split_add2(uint32_t word, float2 (&acc)[kSplitLevels], uint32_t& rem) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
  float2 r = make_float2(__uint_as_float(word << 16), __uint_as_float(word & 0xFFFF0000u));
#pragma unroll
  for (int i = 0; i < kSplitLevels; ++i) {
    const float2 c = make_float2(split_c(i), split_c(i)), nc = make_float2(-split_c(i), -split_c(i));
    const float2 hi = __fadd2_rn(__fadd2_rn(r, c), nc);
    r = __ffma2_rn(hi, m1, r);  // r - hi, exact
    acc[i] = __fadd2_rn(acc[i], hi);
  }
  rem |= __float_as_uint(r.x) | __float_as_uint(r.y);
}

// Pass 1: each CTA reduces kStatsChunk tokens of one (batch, kv head): sums of K (WITH_K) and
// float32 max |V| per channel. A warp reads whole 256-byte rows: lane l handles channels 4l..4l+3,
// warp w tokens w + 8i (128 tokens: the split levels above are exact for 128 values). Each lane's
// sum is the exact sum of its values (levels added smallest first in float64), or, in a CTA that
// met a value the levels do not take, their float64 sum in token order; the 8 warps' partial rows
// are then combined in a fixed order, so the result is deterministic.
template <bool WITH_K>
__global__ void __launch_bounds__(256) kv_stats_partial_kernel(const __nv_bfloat16* __restrict__ k,
                                                               const __nv_bfloat16* __restrict__ v, int Skv, int Hkv,
                                                               int nchunk, double* __restrict__ psum,
                                                               float* __restrict__ pmax) {
  constexpr int kWarps = 8, kTokens = kStatsChunk / kWarps;
  static_assert(kTokens == 128, "128 tokens per lane: the split levels are exact for 128 values");
  __shared__ double ssum[kWarps][kHeadDim];
  __shared__ float smax[kWarps][kHeadDim];
  // The final kernel (which waits for this one) and the Q quantizer behind it may take the SMs this
  // grid's last wave leaves idle.
  pdl_launch_dependents();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __nv_bfloat162 m2[2] = {u32_as_bf162(0u), u32_as_bf162(0u)};  // channel pairs (4l, 4l+1), (4l+2, 4l+3)
  __nv_bfloat162 km2 = u32_as_bf162(0u);                         // max |K| over both pairs
  float2 acc[2][kSplitLevels];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int i = 0; i < kSplitLevels; ++i) acc[p][i] = make_float2(0.0f, 0.0f);
  uint32_t rem = 0u;
  const int j0 = chunk * kStatsChunk + w;
  const int jn = min(Skv, chunk * kStatsChunk + kStatsChunk);
  const size_t row0 = (((size_t)b * Skv + j0) * Hkv + h) * kHeadDim + lane * 4;
  const size_t step = (size_t)kWarps * Hkv * kHeadDim;  // 8 tokens
  for (int i0 = 0; i0 < kTokens && j0 + kWarps * i0 < jn; i0 += kStatsBatch) {
    uint2 kr[kStatsBatch], vr[kStatsBatch];
#pragma unroll
    for (int u = 0; u < kStatsBatch; ++u) {
      kr[u] = vr[u] = make_uint2(0u, 0u);  // zero rows past the end add nothing
      if (j0 + kWarps * (i0 + u) < jn) {
        const size_t off = row0 + (size_t)(i0 + u) * step;
        if constexpr (WITH_K) kr[u] = ld_stream_v2(k + off);
        vr[u] = ld_stream_v2(v + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kStatsBatch; ++u) {
      if constexpr (WITH_K) {
        split_add2(kr[u].x, acc[0], rem);
        split_add2(kr[u].y, acc[1], rem);
        km2 = __hmax2(km2, __hmax2(__habs2(u32_as_bf162(kr[u].x)), __habs2(u32_as_bf162(kr[u].y))));
      }
      // max |V| on bf16 pairs (exact: a max only selects)
      m2[0] = __hmax2(m2[0], __habs2(u32_as_bf162(vr[u].x)));
      m2[1] = __hmax2(m2[1], __habs2(u32_as_bf162(vr[u].y)));
    }
  }
  const float m[4] = {__low2float(m2[0]), __high2float(m2[0]), __low2float(m2[1]), __high2float(m2[1])};
  double s[4] = {0.0, 0.0, 0.0, 0.0};
  if constexpr (WITH_K) {
    // __hmax2 passes over a NaN, whose remainder is NaN and so nonzero
    uint32_t kmax;
    memcpy(&kmax, &km2, sizeof(kmax));
    const bool wide = (rem & 0x7FFFFFFFu) != 0u || (kmax & 0xFFFFu) > (kSplitMaxAbs & 0xFFFFu) ||
                      (kmax >> 16) > (kSplitMaxAbs >> 16);
    if (__syncthreads_or(wide)) {  // rare: this CTA sums its tokens in float64, in token order
      for (int i = 0; i < kTokens && j0 + kWarps * i < jn; ++i) {
        float kf[4];
        bf16x4_to_f32(ld_stream_v2(k + row0 + (size_t)i * step), kf);
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] += (double)kf[e];
      }
    } else {
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        double tx = (double)acc[p][kSplitLevels - 1].x, ty = (double)acc[p][kSplitLevels - 1].y;
#pragma unroll
        for (int i = kSplitLevels - 2; i >= 0; --i) {
          tx += (double)acc[p][i].x;
          ty += (double)acc[p][i].y;
        }
        s[2 * p] = tx;
        s[2 * p + 1] = ty;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if constexpr (WITH_K) ssum[w][lane * 4 + e] = s[e];
    smax[w][lane * 4 + e] = m[e];
  }
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    double a = 0.0;
    float mx = 0.0f;
    for (int r = 0; r < kWarps; ++r) {
      a += ssum[r][threadIdx.x];
      mx = fmaxf(mx, smax[r][threadIdx.x]);
    }
    const size_t o = (((size_t)b * Hkv + h) * nchunk + chunk) * kHeadDim + threadIdx.x;
    if constexpr (WITH_K) psum[o] = a;
    pmax[o] = mx;
  }
}

// Pass 2: combine the chunks of one (batch, kv head) in chunk order, loading eight chunks' partials
// before adding them (the order of the float64 additions is the chunk order all the same).
template <bool WITH_K>
__global__ void __launch_bounds__(128) kv_stats_final_kernel(const double* __restrict__ psum,
                                                             const float* __restrict__ pmax, int Skv, int Hkv,
                                                             int nchunk, float* __restrict__ k_mean,
                                                             float* __restrict__ v_scale) {
  pdl_launch_dependents();  // the Q quantizer reads none of this kernel's inputs or outputs
  pdl_wait();               // the partial sums
  constexpr int kLoads = 8;
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const size_t base = ((size_t)b * Hkv + h) * nchunk * kHeadDim + c;
  double a = 0.0;
  float mx = 0.0f;
  for (int i0 = 0; i0 < nchunk; i0 += kLoads) {
    double ps[kLoads];
    float pm[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const size_t o = base + (size_t)(i0 + u) * kHeadDim;
      ps[u] = (WITH_K && i0 + u < nchunk) ? psum[o] : 0.0;
      pm[u] = (i0 + u < nchunk) ? pmax[o] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      if (i0 + u < nchunk) {
        if constexpr (WITH_K) a += ps[u];
        mx = fmaxf(mx, pm[u]);
      }
    }
  }
  const size_t o = ((size_t)b * Hkv + h) * kHeadDim + c;
  if constexpr (WITH_K) k_mean[o] = __double2float_rn(__ddiv_rn(a, (double)Skv));
  v_scale[o] = __fdiv_rn(mx, 448.0f);
}

// One tensor-wide V scale (QK16PV8 with v_block_size 0): the max of the per-channel scales,
// written back over all of them. Dividing by 448 rounds monotonically, so this equals
// (max |V| over the whole tensor) / 448. One CTA; the array is B * Hkv * 128 floats.
__global__ void __launch_bounds__(1024) v_scale_tensor_kernel(float* __restrict__ v_scale, long long n) {
  __shared__ float red[32];
  float m = 0.0f;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, v_scale[i]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  m = red[0];
  for (long long i = threadIdx.x; i < n; i += blockDim.x) v_scale[i] = m;
}

// E4M3 codes of V / v_scale[b, h, c] (V alone, for QK16PV8): the same arithmetic as the V part of
// the token-block quantizer. A CTA covers kQuantRows tokens of one (batch, kv head); thread t
// keeps channels 8*(t%16).. (and their scales' reciprocals) over tokens t/16 + 16i, loading eight rows
// before it converts any.
__global__ void __launch_bounds__(256) quant_v_kernel(const __nv_bfloat16* __restrict__ v, int Hkv, int Skv,
                                                      const float* __restrict__ v_scale,
                                                      uint8_t* __restrict__ v_codes) {
  pdl_launch_dependents();
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int cg = threadIdx.x & 15, tr = threadIdx.x >> 4;
  const float4* sp = reinterpret_cast<const float4*>(v_scale + ((size_t)b * Hkv + h) * kHeadDim + cg * 8);
  const float4 s0 = sp[0], s1 = sp[1];
  const float vs[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  bool fast[8];
  float rcp[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    fast[e] = scale_in_fast_range(vs[e]);
    rcp[e] = fast[e] ? __frcp_rn(vs[e]) : 0.0f;
  }
  constexpr int kBatch = 8;  // rows loaded before any is converted
  const int j0 = chunk * kQuantRows + tr;
  const int jn = min(Skv, chunk * kQuantRows + kQuantRows);
  const size_t row0 = (((size_t)b * Skv + j0) * Hkv + h) * kHeadDim + cg * 8;
  const size_t step = (size_t)16 * Hkv * kHeadDim;  // 16 tokens
  for (int i0 = 0; i0 < kQuantRows / 16 && j0 + 16 * i0 < jn; i0 += kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (j0 + 16 * (i0 + u) < jn) raw[u] = ld_stream_v4(v + row0 + (size_t)(i0 + u) * step);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (j0 + 16 * (i0 + u) >= jn) break;
      float vf[8];
      bf16x8_to_f32(raw[u], vf);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        if (fast[e] && fast[e + 1]) {
          const float2 v2 = div2_by_scale(make_float2(vf[e], vf[e + 1]), make_float2(vs[e], vs[e + 1]),
                                          make_float2(rcp[e], rcp[e + 1]));
          vf[e] = v2.x;
          vf[e + 1] = v2.y;
        } else {
          vf[e] = quotient(vf[e], vs[e], fast[e], rcp[e]);
          vf[e + 1] = quotient(vf[e + 1], vs[e + 1], fast[e + 1], rcp[e + 1]);
        }
      }
      uint2 w;
      w.x = e4m3x2(vf[0], vf[1]) | (e4m3x2(vf[2], vf[3]) << 16);
      w.y = e4m3x2(vf[4], vf[5]) | (e4m3x2(vf[6], vf[7]) << 16);
      *reinterpret_cast<uint2*>(v_codes + row0 + (size_t)(i0 + u) * step) = w;
    }
  }
  pdl_wait();  // complete only after the kernel before this one
}

// ------------------------------------------------------------------ token-block quantizer
// A CTA covers kQuantRows consecutive tokens of one (batch, head), in warp units of ROWS =
// max(QB, 2) tokens: two rows per iteration, 16 lanes per row (16-byte loads). For QB == 1 each
// half-warp is its own block; otherwise the whole unit is one block. SMOOTH subtracts the K mean.
// A warp takes NU of its units at a time (two units of one or two rows per lane, or one unit of
// eight) and loads all their rows, held as raw bf16, before it reduces any block; the codes are
// then computed from the held rows, so a 16-row block is read once.
template <int QB, int OUT, bool SMOOTH>
__global__ void __launch_bounds__(256) quant_tokens_kernel(const __nv_bfloat16* __restrict__ x, int S, int H,
                                                           const float* __restrict__ mean, void* __restrict__ codes,
                                                           float* __restrict__ scales, int nblk) {
  constexpr int ROWS = QB < 2 ? 2 : QB;
  constexpr int IT = ROWS / 2;               // rows per lane in a unit
  constexpr int UNITS = kQuantRows / ROWS;  // warp units per CTA
  constexpr int PER_WARP = UNITS / 8;
  constexpr int NU = IT >= 8 ? 1 : 2;      // units loaded together
  constexpr float QMAX = (OUT == CODE_E4M3) ? 448.0f : 127.0f;
  static_assert(kQuantRows % 16 == 0 && PER_WARP % NU == 0, "whole blocks per CTA, whole batches per warp");
  pdl_launch_dependents();
  if constexpr (SMOOTH) pdl_wait();  // the mean comes from the kernel before
  const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, cg = lane & 15;
  float mu[8];
  if constexpr (SMOOTH) {
    const float4* mp = reinterpret_cast<const float4*>(mean + ((size_t)b * H + h) * kHeadDim + cg * 8);
    const float4 m0 = mp[0], m1 = mp[1];
    mu[0] = m0.x; mu[1] = m0.y; mu[2] = m0.z; mu[3] = m0.w;
    mu[4] = m1.x; mu[5] = m1.y; mu[6] = m1.z; mu[7] = m1.w;
  }
  auto values = [&](const uint4& raw, float* out) {  // smoothed values of this lane's 8 channels of a row
    bf16x8_to_f32(raw, out);
    if constexpr (SMOOTH) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {  // x - mu as x + (-mu): the same rounding
        const float2 d = __fadd2_rn(make_float2(out[e], out[e + 1]), make_float2(-mu[e], -mu[e + 1]));
        out[e] = d.x;
        out[e + 1] = d.y;
      }
    }
  };
  auto row_offset = [&](int row) { return (((size_t)b * S + row) * H + h) * kHeadDim + cg * 8; };
  for (int t0 = 0; t0 < PER_WARP; t0 += NU) {
    if ((chunk * UNITS + warp + 8 * t0) * ROWS >= S) break;  // later units start later still
    uint4 raw[NU][IT];
#pragma unroll
    for (int n = 0; n < NU; ++n) {
      const int rb = chunk * UNITS + warp + 8 * (t0 + n);
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int row = rb * ROWS + 2 * it + half;
        raw[n][it] = row < S ? ld_stream_v4(x + row_offset(row)) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int n = 0; n < NU; ++n) {
      const int rb = chunk * UNITS + warp + 8 * (t0 + n);  // block of rows (a whole warp unit) within this (b, h)
      if (rb * ROWS >= S) break;                          // the same for every lane of the warp
      float amax = 0.0f;
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        if (rb * ROWS + 2 * it + half >= S) continue;
        float f[8];
        values(raw[n][it], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
      }
      // block absmax: over 16 lanes (QB == 1, one row per half-warp) or the whole warp
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if constexpr (QB > 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
      const float scale = scale_of(amax, QMAX, 1.0f / QMAX);
      const bool fast = scale_in_fast_range(scale);
      const float rcp = fast ? __frcp_rn(scale) : 0.0f;
#pragma unroll
      for (int it = 0; it < IT; ++it) {
        const int row = rb * ROWS + 2 * it + half;
        if (row >= S) continue;
        const size_t off = row_offset(row);
        float q[8];
        values(raw[n][it], q);
        quotients8<OUT != CODE_E4M3>(q, scale, fast, rcp);
        if constexpr (OUT == CODE_E4M3) {
          uint2 w;
          w.x = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
          w.y = e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(codes) + off) = w;
        } else if constexpr (OUT == CODE_I8) {
          const uint2 w = make_uint2(int8_codes4(q[0], q[1], q[2], q[3]), int8_codes4(q[4], q[5], q[6], q[7]));
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(codes) + off) = w;
        } else {  // CODE_I8_AS_F16: the same integer codes, held exactly in fp16
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) w[e] = int8_code_f16x2(q[2 * e], q[2 * e + 1]);
          *reinterpret_cast<uint4*>(static_cast<__half*>(codes) + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // scales: one per block; for QB == 1 lane 0 and lane 16 each own a row (= a block)
      if (QB == 1) {
        const int row = rb * 2 + half;
        if (cg == 0 && row < S) scales[((size_t)b * H + h) * nblk + row] = scale;
      } else if (lane == 0) {
        scales[((size_t)b * H + h) * nblk + rb] = scale;
      }
    }
  }
  pdl_wait();  // complete only after the kernel before this one
}

// ------------------------------------------------------------------ MXFP8 quantizer
// MXFP8 codes of a [B, S, H, 128] BF16 tensor, one E8M0 scale per 32 channels of a token (OCP MX
// v1.0 conversion, as "VisualGen Quantized Attention" names MXFP8 Q/K with blocks of 32 along the
// head dimension): shared exponent e = floor(log2 amax) - 8 clamped to [-127, 127], elements
// E4M3(x / 2^e) rounded to nearest even with saturation. With E the biased float32 exponent of
// amax (0 for zero and subnormals), the stored byte e + 127 is max(E - 8, 0), and x / 2^e is the
// exact product x * 2^(127 - byte) (IEEE multiply, subnormal results kept).
// Four consecutive lanes hold one block (8 channels each, one 16-byte load) and exchange the block
// max with two shuffles; the loop runs per warp, so every shuffle has all 32 lanes.
__global__ void __launch_bounds__(256) mx_quant_kernel(const uint4* __restrict__ x, int S, int H, long long nvec,
                                                       uint2* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long wb = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); wb < nvec; wb += stride) {
    const long long i = wb + lane;  // 16-byte vector: row i / 16 = (b * S + s) * H + h, block (i / 4) % 4
    const bool valid = i < nvec;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid) raw = ld_stream_v4(x + i);
    float f[8];
    bf16x8_to_f32(raw, f);
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const int byte = max((int)(__float_as_uint(a) >> 23) - 8, 0);
    const float mult = __uint_as_float((uint32_t)(254 - byte) << 23);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(f[e], mult);
    uint2 w;
    w.x = e4m3x2(f[0], f[1]) | (e4m3x2(f[2], f[3]) << 16);
    w.y = e4m3x2(f[4], f[5]) | (e4m3x2(f[6], f[7]) << 16);
    if (valid) {
      codes[i] = w;
      if ((lane & 3) == 0) {
        const long long row = i >> 4, t = row / H, s = t % S, b = t / S, h = row % H;
        sf[((b * H + h) * S + s) * 4 + ((i >> 2) & 3)] = (uint8_t)byte;
      }
    }
  }
}

// ------------------------------------------------------------------ NVFP4 quantizer
// NVFP4 ("VisualGen Quantized Attention" names NVFP4 Q/K with blocks of 16 along the head dimension;
// the format is NVIDIA's two-level one): FP4 E2M1 elements, an unsigned E4M3 scale per 16 channels
// of a token, and a float32 tensor scale S = 2688 / amax_T (2688 = 448 * 6). Per block:
// byte = E4M3(float32(amax_b / 6) * S); elements E2M1(float32(x * float32(S / d_b))) with d_b the
// decoded byte (zero codes when d_b = 0). Divisions are IEEE (__fdiv_rn), products single roundings.

// max |x| over a whole tensor, as float32 bits, folded into *amax_bits with atomicMax (float32 bits of
// non-negative values order like the values). *amax_bits must start at 0.
__global__ void __launch_bounds__(256) absmax_kernel(const uint4* __restrict__ x, long long nvec,
                                                     unsigned* __restrict__ amax_bits) {
  float a = 0.0f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (long long)gridDim.x * blockDim.x) {
    float f[8];
    bf16x8_to_f32(ld_stream_v4(x + i), f);
#pragma unroll
    for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) a = fmaxf(a, red[w]);
    atomicMax(amax_bits, __float_as_uint(a));
  }
}

__device__ __forceinline__ float nvfp4_tensor_scale(unsigned amax_bits) {
  const float amax = __uint_as_float(amax_bits);
  return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
}

// value of a non-negative E4M3 byte (bias 7, 3 mantissa bits; exponent field 0 = subnormal, step 2^-9)
__device__ __forceinline__ float e4m3_byte_value(uint32_t b) {
  const uint32_t ex = (b >> 3) & 15u, m = b & 7u;
  return ex == 0 ? (float)m * 0x1p-9f : __uint_as_float(((ex + 120u) << 23) | (m << 20));
}

// two E2M1 codes in one byte: `lo` in bits 0-3, `hi` in bits 4-7 (round to nearest even, saturating)
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two consecutive lanes hold one block (8 channels each, one 16-byte load) and exchange its max
// with one shuffle; the loop runs per warp so every shuffle has all 32 lanes.
__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const uint4* __restrict__ x, int S, int H, long long nvec,
                                                          const unsigned* __restrict__ amax_bits,
                                                          uint32_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const float scale = nvfp4_tensor_scale(*amax_bits);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long wb = (long long)blockIdx.x * blockDim.x + (threadIdx.x & ~31); wb < nvec; wb += stride) {
    const long long i = wb + lane;  // 16-byte vector: row i / 16 = (b * S + s) * H + h, block (i / 2) % 8
    const bool valid = i < nvec;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (valid) raw = ld_stream_v4(x + i);
    float f[8];
    bf16x8_to_f32(raw, f);
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(f[e]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    const uint32_t byte = e4m3x2(__fmul_rn(__fdiv_rn(a, 6.0f), scale), 0.0f) & 0xFFu;
    const float d = e4m3_byte_value(byte);
    const float enc = d > 0.0f ? __fdiv_rn(scale, d) : 0.0f;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) w |= e2m1x2(__fmul_rn(f[2 * e], enc), __fmul_rn(f[2 * e + 1], enc)) << (8 * e);
    if (valid) {
      codes[i] = w;
      if ((lane & 1) == 0) {
        const long long row = i >> 4, t = row / H, s = t % S, b = t / S, h = row % H;
        sf[((b * H + h) * S + s) * 8 + ((i >> 1) & 7)] = (uint8_t)byte;
      }
    }
  }
}

// tensor scales from the two maxima, in place (after every quantizer launch has read them)
__global__ void nvfp4_scales_kernel(unsigned* q_amax_bits, unsigned* k_amax_bits) {
  if (threadIdx.x == 0) {
    if (q_amax_bits != nullptr) *reinterpret_cast<float*>(q_amax_bits) = nvfp4_tensor_scale(*q_amax_bits);
    *reinterpret_cast<float*>(k_amax_bits) = nvfp4_tensor_scale(*k_amax_bits);
  }
}

__global__ void widen_i8_kernel(const int8_t* __restrict__ in, size_t n8, __half* __restrict__ out) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint2 w = *reinterpret_cast<const uint2*>(in + i * 8);
    const int8_t* c = reinterpret_cast<const int8_t*>(&w);
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = (uint32_t)__half_as_ushort(__int2half_rn(c[2 * e])) |
             ((uint32_t)__half_as_ushort(__int2half_rn(c[2 * e + 1])) << 16);
    *reinterpret_cast<uint4*>(out + i * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void zero_i32_kernel(int32_t* p, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = 0;
}

int grid_for(long long work_items, int per_cta) {
  long long g = (work_items + per_cta - 1) / per_cta;
  const long long cap = 152LL * 32;  // a few waves over 152 SMs; the kernels loop beyond that
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

// A launch without dynamic shared memory; pdl adds the programmatic stream serialization attribute
// (see pdl_wait).
template <typename... Params, typename... Args>
cudaError_t launch(void (*kernel)(Params...), dim3 grid, int threads, cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int OUT, bool SMOOTH>
cudaError_t launch_quant_tokens(const void* x, int B, int S, int H, int block, const float* mean, void* codes,
                                float* scales, cudaStream_t stream, bool pdl) {
  const int nblk = (S + block - 1) / block;
  const dim3 grid((S + kQuantRows - 1) / kQuantRows, H, B);
  auto xb = static_cast<const __nv_bfloat16*>(x);
  switch (block) {
    case 1:
      return launch(quant_tokens_kernel<1, OUT, SMOOTH>, grid, 256, stream, pdl, xb, S, H, mean, codes, scales, nblk);
    case 4:
      return launch(quant_tokens_kernel<4, OUT, SMOOTH>, grid, 256, stream, pdl, xb, S, H, mean, codes, scales, nblk);
    case 16:
      return launch(quant_tokens_kernel<16, OUT, SMOOTH>, grid, 256, stream, pdl, xb, S, H, mean, codes, scales,
                    nblk);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_kv_stats(const void* k, const void* v, int B, int Hkv, int Skv, double* psum, float* pmax,
                            float* k_mean, float* v_scale, cudaStream_t stream) {
  const int nchunk = stats_chunks(Skv);
  kv_stats_partial_kernel<true><<<dim3(nchunk, Hkv, B), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(k),
                                                                          static_cast<const __nv_bfloat16*>(v), Skv,
                                                                          Hkv, nchunk, psum, pmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch(kv_stats_final_kernel<true>, dim3(Hkv, B), kHeadDim, stream, true, (const double*)psum,
                (const float*)pmax, Skv, Hkv, nchunk, k_mean, v_scale);
}

cudaError_t launch_v_stats(const void* v, int B, int Hkv, int Skv, float* pmax, float* v_scale, bool per_tensor,
                           cudaStream_t stream) {
  const int nchunk = stats_chunks(Skv);
  kv_stats_partial_kernel<false><<<dim3(nchunk, Hkv, B), 256, 0, stream>>>(
      nullptr, static_cast<const __nv_bfloat16*>(v), Skv, Hkv, nchunk, nullptr, pmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kv_stats_final_kernel<false><<<dim3(Hkv, B), kHeadDim, 0, stream>>>(nullptr, pmax, Skv, Hkv, nchunk, nullptr,
                                                                       v_scale);
  e = cudaGetLastError();
  if (e != cudaSuccess || !per_tensor) return e;
  v_scale_tensor_kernel<<<1, 1024, 0, stream>>>(v_scale, (long long)B * Hkv * kHeadDim);
  return cudaGetLastError();
}

namespace {
cudaError_t quant_v(const void* v, int B, int Hkv, int Skv, const float* v_scale, void* v_codes, cudaStream_t stream,
                    bool pdl) {
  return launch(quant_v_kernel, dim3((Skv + kQuantRows - 1) / kQuantRows, Hkv, B), 256, stream, pdl,
                static_cast<const __nv_bfloat16*>(v), Hkv, Skv, v_scale, static_cast<uint8_t*>(v_codes));
}
}  // namespace

cudaError_t launch_quant_v(const void* v, int B, int Hkv, int Skv, const float* v_scale, void* v_codes,
                           cudaStream_t stream) {
  return quant_v(v, B, Hkv, Skv, v_scale, v_codes, stream, false);
}

cudaError_t launch_quant_q(const void* q, int B, int Hq, int Sq, int q_block, int code_out, void* q_codes,
                           float* q_scale, cudaStream_t stream, bool after_stats) {
  // after launch_kv_stats, Q (which reads none of the statistics) may overlap their final kernel
  switch (code_out) {
    case CODE_I8:
      return launch_quant_tokens<CODE_I8, false>(q, B, Sq, Hq, q_block, nullptr, q_codes, q_scale, stream,
                                                 after_stats);
    case CODE_I8_AS_F16:
      return launch_quant_tokens<CODE_I8_AS_F16, false>(q, B, Sq, Hq, q_block, nullptr, q_codes, q_scale, stream,
                                                        after_stats);
    case CODE_E4M3:
      return launch_quant_tokens<CODE_E4M3, false>(q, B, Sq, Hq, q_block, nullptr, q_codes, q_scale, stream,
                                                   after_stats);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_quant_kv(const void* k, const void* v, int B, int Hkv, int Skv, int k_block, int code_out,
                            const float* k_mean, const float* v_scale, void* k_codes, float* k_scale, void* v_codes,
                            cudaStream_t stream) {
  cudaError_t e = cudaErrorInvalidValue;
  // K by an ordinary launch (everything before it has completed); V, which reads only V and the V
  // scales, may start while K's last CTAs run
  switch (code_out) {
    case CODE_I8:
      e = launch_quant_tokens<CODE_I8, true>(k, B, Skv, Hkv, k_block, k_mean, k_codes, k_scale, stream, false);
      break;
    case CODE_I8_AS_F16:
      e = launch_quant_tokens<CODE_I8_AS_F16, true>(k, B, Skv, Hkv, k_block, k_mean, k_codes, k_scale, stream,
                                                    false);
      break;
    case CODE_E4M3:
      e = launch_quant_tokens<CODE_E4M3, true>(k, B, Skv, Hkv, k_block, k_mean, k_codes, k_scale, stream, false);
      break;
  }
  if (e != cudaSuccess) return e;
  return quant_v(v, B, Hkv, Skv, v_scale, v_codes, stream, true);
}

cudaError_t launch_mx_quant(const void* x, int B, int S, int H, void* codes, uint8_t* sf, cudaStream_t stream) {
  const long long nvec = (long long)B * S * H * (kHeadDim / 8);
  if (nvec == 0) return cudaSuccess;
  mx_quant_kernel<<<grid_for(nvec, 256), 256, 0, stream>>>(static_cast<const uint4*>(x), S, H, nvec,
                                                            static_cast<uint2*>(codes), sf);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_quant(const void* q, const void* k, int B, int Hq, int Hkv, int Sq, int Skv, void* q_codes,
                               void* k_codes, uint8_t* q_sf, uint8_t* k_sf, float* q_scale, float* k_scale,
                               cudaStream_t stream) {
  // q_scale / k_scale first hold the tensors' max |x| (float bits, accumulated from 0), then S
  const long long nq = (long long)B * Sq * Hq * (kHeadDim / 8), nk = (long long)B * Skv * Hkv * (kHeadDim / 8);
  unsigned* qa = reinterpret_cast<unsigned*>(q_scale);
  unsigned* ka = reinterpret_cast<unsigned*>(k_scale);
  cudaError_t e = cudaSuccess;
  if (nq > 0) e = cudaMemsetAsync(qa, 0, sizeof(unsigned), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ka, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  if (nq > 0) absmax_kernel<<<grid_for(nq, 256), 256, 0, stream>>>(static_cast<const uint4*>(q), nq, qa);
  absmax_kernel<<<grid_for(nk, 256), 256, 0, stream>>>(static_cast<const uint4*>(k), nk, ka);
  if (nq > 0)
    nvfp4_quant_kernel<<<grid_for(nq, 256), 256, 0, stream>>>(static_cast<const uint4*>(q), Sq, Hq, nq, qa,
                                                              static_cast<uint32_t*>(q_codes), q_sf);
  nvfp4_quant_kernel<<<grid_for(nk, 256), 256, 0, stream>>>(static_cast<const uint4*>(k), Skv, Hkv, nk, ka,
                                                            static_cast<uint32_t*>(k_codes), k_sf);
  nvfp4_scales_kernel<<<1, 32, 0, stream>>>(nq > 0 ? qa : nullptr, ka);
  return cudaGetLastError();
}

cudaError_t launch_widen_i8(const int8_t* codes, size_t n, void* out_f16, cudaStream_t stream) {
  const size_t n8 = n / 8;  // n is a multiple of 128
  widen_i8_kernel<<<grid_for((long long)n8, 256), 256, 0, stream>>>(codes, n8, static_cast<__half*>(out_f16));
  return cudaGetLastError();
}

cudaError_t launch_zero_i32(int32_t* p, size_t n, cudaStream_t stream) {
  zero_i32_kernel<<<grid_for((long long)n, 256), 256, 0, stream>>>(p, n);
  return cudaGetLastError();
}

}  // namespace ditattn
