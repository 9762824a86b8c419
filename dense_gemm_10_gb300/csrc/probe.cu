// probe.cu -- test support: one tensor-memory-accelerator tile load, issued
// the way the GEMM's producer loads a K-major 16-bit operand tile (128-byte
// swizzle, a box of 64 elements by `rows` rows, completion counted on an
// mbarrier), after which the tile's shared-memory bytes are written back out
// unchanged.  A test compares them with the layout the MMA's shared-memory
// descriptors assume: element (r, c) of the tile at 16-bit position
// r * 64 + (c ^ 8 (r mod 8)), the 16-byte pieces of each 128-byte row permuted
// by the row's index within its group of eight ("[CUDA 优化实战] hgemm sm120 -
// 100KB SMEM 中的“微雕”战争", section 4, the 128B swizzle).
#include <cuda.h>

#include "gemm_internal.h"
#include "ptx.cuh"

namespace g10 {

__global__ void __launch_bounds__(128) tma_tile_probe_kernel(const __grid_constant__ CUtensorMap map, int rows,
                                                             uint16_t* __restrict__ dst, int32_t* status,
                                                             uint64_t wait_limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ int landed;
  // the swizzle pattern repeats every 1024 bytes: the tile starts on such a boundary
  uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(b, static_cast<uint32_t>(rows) * 128u);
    tma_load_3d(smem_u32(tile), &map, b, 0, 0, 0);
    const uint64_t t0 = global_timer_ns();
    bool done = mbar_try_wait(b, 0);
    while (!done && global_timer_ns() - t0 <= wait_limit_ns) done = mbar_try_wait(b, 0);
    if (!done) {
      atomicCAS(status, 0, kStatusTimeout);
      // The copy may still land: wait once more (bounded) before the CTA may
      // exit.  If that wait runs out too, the copy can land after the CTA has
      // left, in shared memory it no longer owns; so a timed-out probe ends its
      // caller's use of probes: the caller reads the status (a stream
      // synchronise) and launches no further probe in the process.
      const uint64_t t1 = global_timer_ns();
      while (!mbar_try_wait(b, 0) && global_timer_ns() - t1 <= wait_limit_ns) {
      }
    }
    landed = done ? 1 : 0;
  }
  __syncthreads();
  if (!landed) return;
  const uint16_t* t = reinterpret_cast<const uint16_t*>(tile);
  for (int i = threadIdx.x; i < rows * 64; i += blockDim.x) dst[i] = t[i];
}

cudaError_t tma_tile_probe_launch(const CUtensorMap& map, int rows, uint16_t* dst, int32_t* status,
                                  uint64_t wait_limit_ns, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(rows) * 128 + 1024;  // the tile plus alignment slack
  tma_tile_probe_kernel<<<1, 128, smem, stream>>>(map, rows, dst, status, wait_limit_ns);
  return cudaGetLastError();
}

}  // namespace g10
