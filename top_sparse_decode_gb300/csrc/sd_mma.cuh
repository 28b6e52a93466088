// Warp-level tensor-core MMA (inline PTX) for the small dense tiles of the
// gather-attend: a KV head's G query rows against 8 or 16 gathered tokens.
#pragma once

#include <stdint.h>

namespace sd {

// d += A B for one m16n8k16 tile, bf16 inputs, fp32 accumulation.  Fragments as the
// PTX ISA lays them out for lane (gid = lane / 4, tig = lane % 4): a0 row gid, cols
// 2tig, 2tig + 1; a1 row gid + 8; a2 / a3 cols + 8; b0 rows 2tig, 2tig + 1 of col
// gid, b1 rows + 8; d0, d1 row gid cols 2tig, 2tig + 1, d2, d3 row gid + 8.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace sd
