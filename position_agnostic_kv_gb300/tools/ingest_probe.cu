// Per-SM shared-memory ingest rate of the copy paths the attention kernels use (a roofline
// calibration, not part of the library): TMA tensor boxes of 16 rows x 64 bf16 columns with
// 128-byte swizzle (the prefill's K/V loads) at ring depths 2/4/6, the same boxes issued half
// per CTA with .multicast::cluster to a 2-CTA cluster, and 1-D bulk copies of whole 4 KB pages
// (the decode's loads).  One CTA per SM; every wait is
// bounded by %globaltimer.  Build and run on the GPU:
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o ingest_probe \
//        position_agnostic_kv_gb300/tools/ingest_probe.cu && ./ingest_probe
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <vector>
#include <cuda.h>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("%s: %s\n", #x, cudaGetErrorString(e)); return 1; } } while (0)

__device__ __forceinline__ uint64_t gtime() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ bool wait_par(uint32_t bar, uint32_t par) {
  const uint64_t t0 = gtime();
  while (true) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(bar), "r"(par) : "memory");
    if (ok) return true;
    if (gtime() - t0 > 1500000000ull) return false;
  }
}
__device__ __forceinline__ uint32_t cluster_rank() { uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr int PAGES = 8, PAGE_BYTES = 4096, STAGE = PAGES * PAGE_BYTES;  // 32 KB stages

// MC = 1: plain loads of all 8 pages; MC = 2: cluster pair, each CTA loads 4 pages multicast to both.
// BULK: one 1-D bulk copy of each whole 4 KB page instead of two tensor boxes (no swizzle).
template <int NST, int MC, bool BULK = false>
__global__ void __launch_bounds__(64, 1) stream(const __grid_constant__ CUtensorMap map, const uint8_t* base,
                                                const int* page_ids, int n_pages_total, int tiles, int* fail) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s0 = (uint32_t(__cvta_generic_to_shared(smem)) + 1023u) & ~1023u;
  const uint32_t bars = s0 + NST * STAGE;  // full[NST], empty[NST]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = MC == 2 ? cluster_rank() : 0;
  const int unit = MC == 2 ? blockIdx.x / 2 : blockIdx.x;  // both CTAs of a pair stream the same pages
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8 * s));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bars + 8 * (NST + s)), "r"(MC));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (MC == 2) cluster_sync(); else __syncthreads();
  if (warp == 0) {  // producer
    for (int j = 0; j < tiles; ++j) {
      const int s = j % NST;
      // a stage is reloaded once every consumer that it lands in (both CTAs with multicast) released it
      if (j >= NST && !wait_par(bars + 8 * (NST + s), ((j / NST) - 1) & 1)) { if (lane == 0) atomicAdd(fail, 1); break; }
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bars + 8 * s), "r"(STAGE) : "memory");
      __syncwarp();
      const int per = PAGES / MC;
      if (lane < per) {
        const int p = int(rank) * per + lane;  // page slot of the stage this CTA issues
        const int pg = page_ids[(unit * 7919 + j * PAGES + p) % n_pages_total];
        const uint32_t dst = s0 + s * STAGE + p * PAGE_BYTES;
        if (BULK)
          asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                       ::"r"(dst), "l"(base + (size_t)pg * PAGE_BYTES), "r"(PAGE_BYTES), "r"(bars + 8 * s) : "memory");
        for (int cb = 0; cb < 2 && !BULK; ++cb) {
          if (MC == 2)
            asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;"
                         ::"r"(dst + cb * 2048), "l"(reinterpret_cast<uint64_t>(&map)), "r"(cb * 64), "r"(pg * 16), "r"(bars + 8 * s), "h"((uint16_t)3) : "memory");
          else
            asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                         ::"r"(dst + cb * 2048), "l"(reinterpret_cast<uint64_t>(&map)), "r"(cb * 64), "r"(pg * 16), "r"(bars + 8 * s) : "memory");
        }
      }
      __syncwarp();
    }
  } else if (lane == 0) {  // consumer: release the stage in this CTA and (multicast) in the peer
    for (int j = 0; j < tiles; ++j) {
      const int s = j % NST;
      if (!wait_par(bars + 8 * s, (j / NST) & 1)) { atomicAdd(fail, 1); break; }
      const uint32_t eb = bars + 8 * (NST + s);
      asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(eb) : "memory");
      if (MC == 2) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(eb), "r"(rank ^ 1u));
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
      }
    }
  }
  if (MC == 2) cluster_sync(); else __syncthreads();
}

// One CTA per SM with P producer warps, each streaming its own NST-stage ring (own barriers)
// and one consumer lane per ring: do several independent rings in one CTA reach the rate of
// several CTAs?
template <int NST, int P>
__global__ void __launch_bounds__(64 * P, 1) stream_multi(const __grid_constant__ CUtensorMap map, const int* page_ids,
                                                          int n_pages_total, int tiles, int* fail) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s0 = (uint32_t(__cvta_generic_to_shared(smem)) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ring = warp >> 1;                       // warps 2r (producer), 2r+1 (consumer)
  const uint32_t rbase = s0 + ring * NST * STAGE;
  const uint32_t bars = s0 + P * NST * STAGE + ring * 2 * NST * 8;
  if (lane == 0 && (warp & 1) == 0) {
    for (int s = 0; s < NST; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8 * s));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8 * (NST + s)));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int unit = blockIdx.x * P + ring;
  if ((warp & 1) == 0) {
    for (int j = 0; j < tiles; ++j) {
      const int s = j % NST;
      if (j >= NST && !wait_par(bars + 8 * (NST + s), ((j / NST) - 1) & 1)) { if (lane == 0) atomicAdd(fail, 1); break; }
      if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bars + 8 * s), "r"(STAGE) : "memory");
      __syncwarp();
      if (lane < PAGES) {
        const int pg = page_ids[(unit * 7919 + j * PAGES + lane) % n_pages_total];
        const uint32_t dst = rbase + s * STAGE + lane * PAGE_BYTES;
        for (int cb = 0; cb < 2; ++cb)
          asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                       ::"r"(dst + cb * 2048), "l"(reinterpret_cast<uint64_t>(&map)), "r"(cb * 64), "r"(pg * 16), "r"(bars + 8 * s) : "memory");
      }
      __syncwarp();
    }
  } else if (lane == 0) {
    for (int j = 0; j < tiles; ++j) {
      const int s = j % NST;
      if (!wait_par(bars + 8 * s, (j / NST) & 1)) { atomicAdd(fail, 1); break; }
      asm volatile("mbarrier.arrive.release.cluster.shared::cta.b64 _, [%0];" ::"r"(bars + 8 * (NST + s)) : "memory");
    }
  }
  __syncthreads();
}

template <int NST, int P>
int run_multi(const CUtensorMap& map, const int* ids, int n_pages, int grid, int tiles, int* fail) {
  auto kern = stream_multi<NST, P>;
  const int smem = P * NST * STAGE + P * 2 * NST * 8 + 1024;
  CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  float best = 1e30f;
  for (int rep = 0; rep < 3; ++rep) {
    cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
    cudaEventRecord(a);
    kern<<<grid, 64 * P, smem>>>(map, ids, n_pages, tiles, fail);
    cudaEventRecord(b); CK(cudaEventSynchronize(b)); CK(cudaGetLastError());
    float ms; cudaEventElapsedTime(&ms, a, b); if (ms < best) best = ms;
  }
  int f; CK(cudaMemcpy(&f, fail, 4, cudaMemcpyDeviceToHost));
  const double arrived = (double)grid * P * tiles * STAGE;
  printf("tma-%d-rings/CTA NST %d grid %3d: %8.1f us  arriving per SM %6.1f GB/s  fetched total %7.1f GB/s  fail %d\n", P, NST,
         grid, best * 1e3, arrived / best / 1e6 / grid, arrived / best / 1e6, f);
  return 0;
}

typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int g_sms = 0;  // SM count: "per SM" divides by min(grid, SMs) (grids above it put 2 CTAs on an SM)

template <int NST, int MC, bool BULK = false>
int run(const CUtensorMap& map, const uint8_t* base, const int* ids, int n_pages, int grid, int tiles, int* fail,
        const char* name) {
  auto kern = stream<NST, MC, BULK>;
  const int smem = NST * STAGE + 2 * NST * 8 + 1024;
  CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid); cfg.blockDim = dim3(64); cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = MC; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  cfg.attrs = at; cfg.numAttrs = 1;
  float best = 1e30f;
  for (int rep = 0; rep < 3; ++rep) {
    cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
    cudaEventRecord(a);
    CK(cudaLaunchKernelEx(&cfg, kern, map, base, ids, n_pages, tiles, fail));
    cudaEventRecord(b); CK(cudaEventSynchronize(b)); CK(cudaGetLastError());
    float ms; cudaEventElapsedTime(&ms, a, b); if (ms < best) best = ms;
  }
  int f; CK(cudaMemcpy(&f, fail, 4, cudaMemcpyDeviceToHost));
  const double arrived = (double)grid * tiles * STAGE;  // bytes landing in shared memory, all CTAs
  const int sms_used = grid < g_sms ? grid : g_sms;
  printf("%-14s NST %d grid %3d: %8.1f us  arriving per SM %6.1f GB/s  fetched total %7.1f GB/s  fail %d\n", name, NST, grid,
         best * 1e3, arrived / best / 1e6 / sms_used, arrived / MC / best / 1e6, f);
  return 0;
}

int main() {
  int sms = 0; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  g_sms = sms;
  const int n_pages = 1 << 18;
  uint8_t* buf; CK(cudaMalloc(&buf, (size_t)n_pages * PAGE_BYTES));
  CK(cudaMemset(buf, 1, (size_t)n_pages * PAGE_BYTES));
  std::vector<int> ids(n_pages);
  for (int i = 0; i < n_pages; ++i) ids[i] = i;
  srand(1); for (int i = n_pages - 1; i > 0; --i) { int k = rand() % (i + 1); std::swap(ids[i], ids[k]); }
  int* d_ids; CK(cudaMalloc(&d_ids, n_pages * sizeof(int)));
  CK(cudaMemcpy(d_ids, ids.data(), n_pages * sizeof(int), cudaMemcpyHostToDevice));
  int* fail; CK(cudaMalloc(&fail, 4)); CK(cudaMemset(fail, 0, 4));
  void* fp = nullptr; cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault, &q));
  CUtensorMap map;
  const cuuint64_t dims[2] = {128, (cuuint64_t)n_pages * 16}, strides[1] = {256};
  const cuuint32_t box[2] = {64, 16}, es[2] = {1, 1};
  if (((EncFn)fp)(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    printf("encode failed\n"); return 1;
  }
  const int tiles = 400;
  for (int grid : {16, 64, 128, 152}) {
    if (run<2, 1>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma")) return 1;
    if (run<4, 1>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma")) return 1;
    if (run<6, 1>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma")) return 1;
    if (run<2, 2>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma-multicast")) return 1;
    if (run<4, 2>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma-multicast")) return 1;
    if (run<4, 1, true>(map, buf, d_ids, n_pages, grid, tiles, fail, "bulk-4KB")) return 1;
  }
  // one CTA per SM with two or three independent rings (producer warp + barriers each)
  if (run_multi<3, 2>(map, d_ids, n_pages, sms, tiles, fail)) return 1;
  if (run_multi<2, 3>(map, d_ids, n_pages, sms, tiles, fail)) return 1;
  // two CTAs per SM (each with half the ring): does the rate per SM grow with issuing CTAs?
  {
    const int grid = 2 * sms;
    if (run<2, 1>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma-2cta/SM")) return 1;
    if (run<3, 1>(map, buf, d_ids, n_pages, grid, tiles, fail, "tma-2cta/SM")) return 1;
    if (run<3, 1, true>(map, buf, d_ids, n_pages, grid, tiles, fail, "bulk-2cta/SM")) return 1;
  }
  return 0;
}
