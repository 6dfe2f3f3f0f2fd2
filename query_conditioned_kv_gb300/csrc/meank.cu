// meank.cu — Mean-K index build (KVMem, "Query-conditioned retrieval": one
// RoPE-stripped mean key per layer, KV head and 32-token block).
//
// One thread owns 8 consecutive head-dim elements of one output block row
// and walks the block's 32 tokens with 16-byte loads; the D/8 threads of a
// block row read each 2·D-byte token row as one coalesced segment.  The sum
// is kept in fp64 (exact for 32 bf16 values whose magnitudes span < 2^40),
// divided by 32 (exact) and rounded once to bf16 with __double2bfloat16
// (round to nearest even) — the result equals the exact mean rounded once.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void __launch_bounds__(256)
k_build_meank(const uint16_t *__restrict__ kraw, uint16_t *__restrict__ meank,
              int64_t n_out_chunks, int64_t nb, int chunks_per_row) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_out_chunks) return;
  int64_t row_blk = t / chunks_per_row;  // (row, block)
  int c = (int)(t - row_blk * chunks_per_row);
  const int D = chunks_per_row * 8;
  const uint16_t *src = kraw + row_blk * (int64_t)kBlock * D + c * 8;
  double acc[8];
#pragma unroll
  for (int e = 0; e < 8; e++) acc[e] = 0.0;
#pragma unroll 8
  for (int tok = 0; tok < kBlock; tok++) {
    uint4 v = ld_stream(src + (int64_t)tok * D);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
      acc[2 * e] += (double)bf16_lo(w[e]);
      acc[2 * e + 1] += (double)bf16_hi(w[e]);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; e++) {
    __nv_bfloat16 lo = __double2bfloat16(acc[2 * e] * (1.0 / kBlock));
    __nv_bfloat16 hi = __double2bfloat16(acc[2 * e + 1] * (1.0 / kBlock));
    o[e] = (uint32_t)(*reinterpret_cast<uint16_t *>(&lo)) |
           ((uint32_t)(*reinterpret_cast<uint16_t *>(&hi)) << 16);
  }
  (void)nb;
  *reinterpret_cast<uint4 *>(meank + row_blk * D + c * 8) =
      make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_build_meank(const uint16_t *kraw, uint16_t *meank,
                               int64_t rows, int64_t n_tok, int D,
                               cudaStream_t s) {
  int64_t nb = n_tok / kBlock;
  int cpr = D / 8;
  int64_t n = rows * nb * cpr;
  int64_t grid = (n + 255) / 256;
  k_build_meank<<<(unsigned)grid, 256, 0, s>>>(kraw, meank, n, nb, cpr);
  return cudaGetLastError();
}

}  // namespace kvc
