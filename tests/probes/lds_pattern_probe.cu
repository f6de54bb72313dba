// Standalone probe (test infrastructure, not part of the library): SM cycles per warp-wide shared
// memory load for the access patterns a four-lanes-per-channel recurrence can use.  Each kernel:
// 12 warps per CTA, one CTA per SM, every warp issuing ITER loads of one pattern over a 32-step
// table of 64-byte rows and accumulating the values (so the loads are kept); thread 0 records the
// clock cycles.  Under ncu, l1tex__data_pipe_lsu_wavefronts_mem_shared_op_ld.sum divided by
// smsp__sass_inst_executed_op_shared_ld.sum gives the wavefronts per load instruction.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA error %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

constexpr int ITER = 4096, WARPS = 12, T = 32;

template <int P>
__global__ void __launch_bounds__(WARPS * 32) lds_kernel(float* out, long long* cyc) {
  __shared__ __align__(16) float Bs[T * 20];
  for (int i = threadIdx.x; i < T * 20; i += blockDim.x) Bs[i] = 0.001f * i;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  float4 acc = make_float4(0, 0, 0, 0);
  const long long t0 = clock64();
#pragma unroll 8
  for (int it = 0; it < ITER; ++it) {
    const int t = it & (T - 1);
    float4 v;
    if constexpr (P == 0) {  // quarter-uniform: g = lane / 8, LDS.128 of B[t][4g..4g+3]
      v = *reinterpret_cast<const float4*>(Bs + t * 20 + 4 * (lane >> 3));
    } else if constexpr (P == 1) {  // g = lane % 4: each quarter reads the whole 64-byte row
      v = *reinterpret_cast<const float4*>(Bs + t * 20 + 4 * (lane & 3));
    } else if constexpr (P == 2) {  // warp-uniform LDS.128
      v = *reinterpret_cast<const float4*>(Bs + t * 20);
    } else if constexpr (P == 4) {  // step-table style LDS.64: 8 distinct addresses (lane % 8), stride 68 words
      const float2 a = *reinterpret_cast<const float2*>(Bs + ((lane & 7) * 68 + 2 * t) % (T * 20 - 2));
      v = make_float4(a.x, a.y, 0, 0);
    } else if constexpr (P == 5) {  // the same with 4 consecutive lanes sharing an address (lane / 4)
      const float2 a = *reinterpret_cast<const float2*>(Bs + ((lane >> 2) * 68 + 2 * t) % (T * 20 - 2));
      v = make_float4(a.x, a.y, 0, 0);
    }
    acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
  }
  const long long t1 = clock64();
  if (acc.x + acc.y + acc.z + acc.w == 1234.5f) out[threadIdx.x] = acc.x;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

template <int P>
int run(const char* name, float* out, long long* cyc, int sms) {
  for (int r = 0; r < 2; ++r) {
    lds_kernel<P><<<sms, WARPS * 32>>>(out, cyc);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
  }
  long long h[256];
  CK(cudaMemcpy(h, cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost));
  double m = 0;
  for (int i = 0; i < sms; ++i) m += h[i];
  m /= sms;
  printf("%-44s %6.2f cycles per warp-load-instruction per SM\n", name, m / (double(ITER) * WARPS));
  return 0;
}

int main() {
  int sms;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  float* out;
  long long* cyc;
  CK(cudaMalloc(&out, 4096 * 4));
  CK(cudaMalloc(&cyc, 256 * 8));
  if (run<0>("LDS.128 quarter-uniform (g = lane/8)", out, cyc, sms)) return 1;
  if (run<1>("LDS.128 row per quarter (g = lane%4)", out, cyc, sms)) return 1;
  if (run<2>("LDS.128 warp-uniform", out, cyc, sms)) return 1;
  if (run<4>("LDS.64 8 distinct (lane%8)", out, cyc, sms)) return 1;
  if (run<5>("LDS.64 8 distinct (lane/4)", out, cyc, sms)) return 1;
  printf("done\n");
  return 0;
}
