// Test probe (built by tests/test_gpu_division.py): compares the prepass's reciprocal-based
// division (scalar and packed) with IEEE division (__fdiv_rn) bit for bit, for every quotient the
// quantizers can form (|x / s| <= 448) that can change a code (|x / s| >= 2^-12); for the smaller
// ones, which encode to a signed zero, it checks the sign and that they stay below 2^-11. The
// packed form without the sign of zero (INT8 codes only) is checked on the first range. It also
// checks the block scales amax / qmax for every float32 block max.
#include <cuda_runtime.h>

#include "../../diffusion_transformer_attention_gb300/csrc/quant_math.cuh"

__global__ void div_check_kernel(const float* xs, long long nx, const float* ss, int ns, unsigned long long* bad,
                                 unsigned long long* checked, float* samples) {
  unsigned long long nb = 0, nc = 0;
  const long long total = nx * ns;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const float x = xs[i % nx], s = ss[i / nx];
    if (!ditattn::scale_in_fast_range(s)) continue;
    const float ref = __fdiv_rn(x, s);
    if (!(fabsf(ref) <= 448.0f)) continue;  // quotients the quantizers form: |x| <= absmax = s * QMAX
    ++nc;
    const float r = __frcp_rn(s);
    const float q = ditattn::div_by_scale(x, s, r);
    // the packed forms, with x and -x in their two lanes
    const float2 q2 = ditattn::div2_by_scale(make_float2(x, -x), make_float2(s, s), make_float2(r, r));
    const float2 q3 = ditattn::div2_by_scale<false>(make_float2(x, -x), make_float2(s, s), make_float2(r, r));
    bool ok;
    if (fabsf(ref) >= 0x1p-12f) {  // can change a code: equal bit for bit
      ok = __float_as_uint(q) == __float_as_uint(ref) && __float_as_uint(q2.x) == __float_as_uint(ref) &&
           __float_as_uint(q2.y) == __float_as_uint(-ref) && __float_as_uint(q3.x) == __float_as_uint(ref) &&
           __float_as_uint(q3.y) == __float_as_uint(-ref);
    } else {  // a zero code: its sign, and a magnitude that encodes to zero
      const bool neg = signbit(ref);
      ok = (bool)signbit(q) == neg && (bool)signbit(q2.x) == neg && (bool)signbit(q2.y) == !neg &&
           fabsf(q) < 0x1p-11f && fabsf(q2.x) < 0x1p-11f && fabsf(q2.y) < 0x1p-11f && fabsf(q3.x) < 0x1p-11f &&
           fabsf(q3.y) < 0x1p-11f;
    }
    if (!ok) {
      ++nb;
      const unsigned long long slot = atomicAdd(bad + 1, 1ull);  // bad[1]: samples taken so far
      if (slot < 8) {
        samples[4 * slot] = x;
        samples[4 * slot + 1] = s;
        samples[4 * slot + 2] = q;
        samples[4 * slot + 3] = ref;
      }
    }
  }
  atomicAdd(bad, nb);
  atomicAdd(checked, nc);
}

// The block scales: scale_of(amax, qmax) against amax / qmax for qmax 127 and 448, over |x| for
// every x (a block max is any non-negative float32: a bf16 value, or a smoothed K value).
__global__ void scale_check_kernel(const float* xs, long long nx, unsigned long long* bad, unsigned long long* checked) {
  unsigned long long nb = 0, nc = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nx; i += (long long)gridDim.x * blockDim.x) {
    const float a = fabsf(xs[i]);
    if (!isfinite(a)) continue;
    nc += 2;
    if (__float_as_uint(ditattn::scale_of(a, 127.0f, 1.0f / 127.0f)) != __float_as_uint(__fdiv_rn(a, 127.0f))) ++nb;
    if (__float_as_uint(ditattn::scale_of(a, 448.0f, 1.0f / 448.0f)) != __float_as_uint(__fdiv_rn(a, 448.0f))) ++nb;
  }
  atomicAdd(bad, nb);
  atomicAdd(checked, nc);
}

// result_host[0] = mismatches, [1] = values checked.
extern "C" int scale_check(const float* xs_host, long long nx, unsigned long long* result_host) {
  float* xs = nullptr;
  unsigned long long* res = nullptr;
  if (cudaMalloc(&xs, nx * sizeof(float)) != cudaSuccess) return 1;
  if (cudaMalloc(&res, 2 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  cudaMemcpy(xs, xs_host, nx * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemset(res, 0, 2 * sizeof(unsigned long long));
  scale_check_kernel<<<152 * 8, 256>>>(xs, nx, res, res + 1);
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(result_host, res, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaFree(xs);
  cudaFree(res);
  return e == cudaSuccess ? 0 : 2;
}

// result_host[0] = mismatches, [2] = quotients checked; samples_host: up to 8 (x, s, q, ref) rows.
extern "C" int div_check(const float* xs_host, long long nx, const float* ss_host, int ns,
                         unsigned long long* result_host, float* samples_host) {
  float *xs = nullptr, *ss = nullptr, *smp = nullptr;
  unsigned long long* res = nullptr;
  if (cudaMalloc(&xs, nx * sizeof(float)) != cudaSuccess) return 1;
  if (cudaMalloc(&ss, ns * sizeof(float)) != cudaSuccess) return 1;
  if (cudaMalloc(&smp, 32 * sizeof(float)) != cudaSuccess) return 1;
  if (cudaMalloc(&res, 3 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  cudaMemcpy(xs, xs_host, nx * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemcpy(ss, ss_host, ns * sizeof(float), cudaMemcpyHostToDevice);
  cudaMemset(res, 0, 3 * sizeof(unsigned long long));
  cudaMemset(smp, 0, 32 * sizeof(float));
  div_check_kernel<<<152 * 8, 256>>>(xs, nx, ss, ns, res, res + 2, smp);
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(result_host, res, 3 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaMemcpy(samples_host, smp, 32 * sizeof(float), cudaMemcpyDeviceToHost);
  cudaFree(xs);
  cudaFree(ss);
  cudaFree(smp);
  cudaFree(res);
  return e == cudaSuccess ? 0 : 2;
}
