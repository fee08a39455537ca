// Q4_0 with interleaved nibbles (LQ_FMT_Q4_0I): the order the pages' Q4
// kernels read, gemv_q4_decode and gemm_q4 (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs), where byte j of a block holds element 2j in
// its low nibble and element 2j+1 in its high nibble.
//
// The library's Q4_0 kernels pair the low nibble of byte j with activation
// j of the block and the high nibble with activation 16+j. Feeding them the
// block's activations reordered, even elements first (element 2j to slot j)
// and odd ones after (element 2j+1 to slot 16+j), makes them compute
// sum_j q_2j a_2j + q_2j+1 a_2j+1, the interleaved product: the weight bytes
// stay as they are and only A, which every kernel already rearranges once,
// is stored in another order.
#pragma once
#include <cstdint>

namespace lq {
namespace q4i {

// Slot of element e (0..31) of a block.
__host__ __device__ constexpr int slot_of(int e) { return (e & 1) ? 16 + (e >> 1) : (e >> 1); }

// Stores the 16-byte chunk i (elements 4i .. 4i+3 of a block, as loaded) at
// the slots the standard-order kernels read, given the shared-memory address
// of the block's 32 floats: elements 4i and 4i+2 go to slots 2i and 2i+1,
// elements 4i+1 and 4i+3 to slots 16+2i and 17+2i.
__device__ __forceinline__ void store_chunk(uint32_t block_addr, int i, uint4 v) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(block_addr + 8u * i), "r"(v.x), "r"(v.z) : "memory");
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(block_addr + 64u + 8u * i), "r"(v.y), "r"(v.w)
               : "memory");
}

}  // namespace q4i
}  // namespace lq
