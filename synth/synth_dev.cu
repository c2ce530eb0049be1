// synth_dev.cu — device fill of MX-quantised expert matrices from synth.h.
//
// The same counter-based definition as the host fill (synth_host.c), run on
// the GPU so that hundreds of experts (tens of GB) can be made in HBM in
// milliseconds.  Input bytes only: nothing here is part of the MoE layer.
// Built with --fmad=false so that no multiply-add is contracted.
#include <cuda_runtime.h>

#include "synth.h"

namespace {

__global__ void syn_fill_mx_kernel(uint64_t key, int64_t rows, int64_t cols, uint8_t* q, uint8_t* s) {
  const int64_t nb = cols / 32;
  const int64_t nblocks = rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / nb, b = i % nb;
    uint8_t qb[16];
    uint8_t sb;
    syn_mx_block(key, cols, r, b, qb, &sb);
    // Both sides are 16-byte aligned (row pitch cols/2 is a multiple of 16).
    uint4 v;
    v.x = (uint32_t)qb[0] | ((uint32_t)qb[1] << 8) | ((uint32_t)qb[2] << 16) | ((uint32_t)qb[3] << 24);
    v.y = (uint32_t)qb[4] | ((uint32_t)qb[5] << 8) | ((uint32_t)qb[6] << 16) | ((uint32_t)qb[7] << 24);
    v.z = (uint32_t)qb[8] | ((uint32_t)qb[9] << 8) | ((uint32_t)qb[10] << 16) | ((uint32_t)qb[11] << 24);
    v.w = (uint32_t)qb[12] | ((uint32_t)qb[13] << 8) | ((uint32_t)qb[14] << 16) | ((uint32_t)qb[15] << 24);
    *reinterpret_cast<uint4*>(q + r * (cols / 2) + b * 16) = v;
    s[r * nb + b] = sb;
  }
}

}  // namespace

// Fill q [rows][cols/2] and s [rows][cols/32] (device pointers, q 16-byte
// aligned, cols % 32 == 0) on the given stream.  Returns a cudaError_t value.
extern "C" int syn_dev_fill_mx(uint64_t key, int64_t rows, int64_t cols, void* q, void* s, void* stream) {
  if (cols % 32 != 0 || rows < 0) return (int)cudaErrorInvalidValue;
  if (((uintptr_t)q & 15u) != 0) return (int)cudaErrorInvalidValue;
  const int64_t nblocks = rows * (cols / 32);
  if (nblocks == 0) return 0;
  int64_t grid = (nblocks + 255) / 256;
  if (grid > 152 * 64) grid = 152 * 64;
  syn_fill_mx_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(key, rows, cols, (uint8_t*)q, (uint8_t*)s);
  return (int)cudaGetLastError();
}
