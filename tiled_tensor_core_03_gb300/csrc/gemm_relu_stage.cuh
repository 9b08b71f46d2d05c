// gemm_relu_stage.cuh -- copies of operands whose rows TMA cannot describe.
//
// TMA needs every row of a matrix to start on a 16-byte boundary, so a
// row-major fp16 matrix whose column count is not a multiple of 8 (or whose
// base is not 16-byte aligned) cannot be loaded by the TMA kernels.  The
// predicated-load kernel handles such operands inside the GEMM, re-shifting
// every row segment each time a tile reads it: A once per column of tiles,
// B once per row of tiles.  Given scratch memory, the library instead copies
// each such operand once into rows of pitch round_up(cols, 8) elements at a
// 16-byte-aligned address, and the TMA kernel reads the copy (its tensor map
// keeps the true column count, so TMA zero-fills the columns past it).
//
// One thread per 16-byte chunk of a copied row: it reads the one or two
// aligned 16-byte blocks of the source that hold the chunk's eight elements
// (never a block past the row's last element, so never past the matrix),
// shifts them into place and stores the chunk with one 16-byte store; the
// pad elements of a row's last chunk are written as zeros.  Consecutive
// threads take consecutive chunks of a row, so loads and stores coalesce.
#pragma once

#include "gemm_relu_kernels.cuh"

namespace gemmrelu {
namespace stage {

using namespace sm103;

// One matrix to copy: rows x cols at `src` (2-byte aligned) into `dst`
// (16-byte aligned) with row pitch `pitch` = round_up(cols, 8) elements.
struct Job {
    const uint16_t *src;
    uint16_t *dst;
    int64_t rows, cols, pitch;
};

// Up to two matrices (A and B of one GEMM) in one launch: chunks
// [0, chunks0) belong to job 0, the rest to job 1.
struct Params {
    Job job[2];
    int64_t chunks0, total;
};

__global__ void __launch_bounds__(256) stage_rows_kernel(const Params p) {
    pdl_wait_primary();       // the operands may come from the previous grid
    pdl_launch_dependents();  // the GEMM's set-up may overlap this copy
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < p.total; g += step) {
        const bool second = g >= p.chunks0;
        const Job &j = second ? p.job[1] : p.job[0];
        const int64_t idx = second ? g - p.chunks0 : g;
        const int64_t per_row = j.pitch / 8;
        const int64_t row = idx / per_row;
        const int64_t e0 = 8 * (idx - row * per_row);
        const int nvalid = (int)(j.cols - e0 < 8 ? j.cols - e0 : 8);
        const uintptr_t addr = reinterpret_cast<uintptr_t>(j.src + row * j.cols + e0);
        const uint32_t off = (uint32_t)(addr & 15u);
        const uint4 *blk = reinterpret_cast<const uint4 *>(addr - off);
        const uint4 v0 = __ldg(blk);
        // the second block only when the chunk's last element lies in it
        const uint4 v1 = off + 2u * (uint32_t)nvalid > 16u ? __ldg(blk + 1) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 v = keep_first(window16(v0, v1, make_shift(off)), nvalid);
        *reinterpret_cast<uint4 *>(j.dst + row * j.pitch + e0) = v;
    }
}

}  // namespace stage
}  // namespace gemmrelu
