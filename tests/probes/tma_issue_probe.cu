// Standalone probe (test infrastructure, not part of the library): how long issuing 2-D tensor
// copies (cp.async.bulk.tensor) takes the issuing thread on this GPU, and when the copies land.
// One CTA per SM (or one CTA in all) issues K = 16 copies of a bf16 box into shared memory, from
// one thread or spread over four warps, with the tensor map in the kernel's parameter space or in
// global memory; thread 0 waits (bounded) on the mbarrier that counts the bytes.  Prints, per
// case, the issuing threads' cycles and the cycles until every copy had landed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdio>
#include <cstdint>
#include <vector>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA error %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ CUtensorMap g_map;

struct Maps { CUtensorMap m; };

constexpr int K = 16;           // copies per issuing thread
constexpr int L = 2048;
constexpr int ROWS = 148 * 128;
constexpr long long kLimit = 1LL << 30;

template <int BOXR, bool GLOBAL_MAP, int ISSUERS>
__global__ void __launch_bounds__(128) probe(const __grid_constant__ Maps maps, long long* out) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ long long t_issue[4], t_done;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kBox = 32 * BOXR * 2;
  unsigned char* buf = smem + ((128u - (su32(smem) & 127u)) & 127u);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&bar)), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const void* map = GLOBAL_MAP ? static_cast<const void*>(&g_map) : static_cast<const void*>(&maps.m);
  if (tid == 0)
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&bar)),
                 "r"(uint32_t(K * kBox)) : "memory");
  __syncthreads();
  const long long t0 = clock64();
  if (lane == 0 && warp < ISSUERS) {
    for (int i = warp; i < K; i += ISSUERS) {
      const int row = (blockIdx.x * 128 + (i * BOXR) % 128);
      const int x = 32 * (i / (128 / BOXR));
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(su32(buf + i * kBox)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(su32(&bar))
          : "memory");
    }
    t_issue[warp] = clock64() - t0;
  }
  if (tid == 0) {
    uint32_t done = 0;
    long long spins = 0;
    while (!done && clock64() - t0 < kLimit) {
      asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
                   " selp.u32 %0, 1, 0, p;\n}\n" : "=r"(done) : "r"(su32(&bar)), "r"(0u) : "memory");
      ++spins;
    }
    t_done = done ? clock64() - t0 : -1;
  }
  __syncthreads();
  if (tid == 0) {
    long long mx = 0;
    for (int w = 0; w < ISSUERS; ++w) mx = t_issue[w] > mx ? t_issue[w] : mx;
    out[blockIdx.x * 2] = mx;
    out[blockIdx.x * 2 + 1] = t_done;
  }
}

template <int BOXR, bool G, int IS>
int run(const char* name, PFN_cuTensorMapEncodeTiled_v12000 enc, void* base, long long* dout, int ctas) {
  Maps maps;
  const cuuint64_t dims[2] = {L, ROWS};
  const cuuint64_t strides[1] = {L * 2};
  const cuuint32_t box[2] = {32, BOXR};
  const cuuint32_t el[2] = {1, 1};
  if (enc(&maps.m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    printf("encode failed\n");
    return 1;
  }
  CK(cudaMemcpyToSymbol(g_map, &maps.m, sizeof(CUtensorMap)));
  const int smem = K * 32 * BOXR * 2 + 128;
  auto k = probe<BOXR, G, IS>;
  CK(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  std::vector<long long> h(ctas * 2);
  for (int rep = 0; rep < 3; ++rep) {
    k<<<ctas, 128, smem>>>(maps, dout);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
  }
  CK(cudaMemcpy(h.data(), dout, ctas * 2 * sizeof(long long), cudaMemcpyDeviceToHost));
  double is = 0, dn = 0;
  int bad = 0;
  for (int i = 0; i < ctas; ++i) { is += h[2 * i]; if (h[2 * i + 1] < 0) ++bad; else dn += h[2 * i + 1]; }
  printf("%-34s ctas %3d  issue %7.0f cyc (%5.0f per copy per issuer)  all landed %7.0f cyc  timeouts %d\n", name, ctas,
         is / ctas, is / ctas / (K / IS), dn / ctas, bad);
  return 0;
}

int main() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  void* base;
  CK(cudaMalloc(&base, size_t(ROWS) * L * 2));
  CK(cudaMemset(base, 0, size_t(ROWS) * L * 2));
  long long* dout;
  CK(cudaMalloc(&dout, 148 * 2 * sizeof(long long)));
  for (int ctas : {1, 148}) {
    if (run<32, false, 1>("box32 param 1 issuer", enc, base, dout, ctas)) return 1;
    if (run<32, true, 1>("box32 global 1 issuer", enc, base, dout, ctas)) return 1;
    if (run<8, false, 1>("box8 param 1 issuer", enc, base, dout, ctas)) return 1;
    if (run<32, false, 4>("box32 param 4 issuers", enc, base, dout, ctas)) return 1;
  }
  printf("done\n");
  return 0;
}
