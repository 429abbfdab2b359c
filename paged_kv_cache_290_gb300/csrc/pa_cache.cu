// KV scatter-write: put this step's new K/V tokens into their paged-cache slots.
//
// "vLLM: LLM Inference That Doesn't Waste Your GPU", "KV cache, in one picture": each processed
// token's K/V is stored once and reused by every later token; "Local_LLM_03_vLLM_Architecture",
// paged-KV slide: that store is a pool of fixed-size blocks.  Token t with slot = blk*bs + off
// goes to k_cache[blk][h][off][:] for every kv head h (pool layout [NB][Hkv][bs][d]).
//
// One thread moves one 16-byte chunk of K and the matching chunk of V; consecutive threads
// cover consecutive chunks of a (token, head) row, so both the reads and the writes of a row are
// full 128-byte-line transactions.  fp16 cache: a pure copy, the cache receives the exact bit
// patterns.  FP8 cache: a chunk is 16 codes, each the E4M3 code of x * (1/scale) (float32).
#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const CacheArgs a) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per (token, head) row
  // The attention kernel that follows is a programmatic dependent: let it start setting up
  // now; it waits for this grid to finish (griddepcontrol.wait) before reading anything.
  grid_launch_dependents();
  const int64_t total = a.num_tokens * a.num_kv_heads * kChunks;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ch = static_cast<int>(idx % kChunks);
    const int64_t row = idx / kChunks;
    const int h = static_cast<int>(row % a.num_kv_heads);
    const int64_t t = row / a.num_kv_heads;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= a.num_blocks * a.block_size) {
      atomicOr(a.err, kErrSlotRange);
      continue;
    }
    const int64_t blk = slot / a.block_size;
    const int64_t off = slot % a.block_size;
    const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * D + ch * 8;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(a.k + t * a.k_stride + h * D + ch * 8));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(a.v + t * a.v_stride + h * D + ch * 8));
    *reinterpret_cast<uint4*>(static_cast<__half*>(a.k_cache) + dst) = kv;
    *reinterpret_cast<uint4*>(static_cast<__half*>(a.v_cache) + dst) = vv;
  }
}

// 16 fp16 values (two 16-byte loads) -> 16 E4M3 codes of x * inv.
__device__ __forceinline__ uint4 quantize16(const __half* src, float inv) {
  const uint4 lo = __ldg(reinterpret_cast<const uint4*>(src));
  const uint4 hi = __ldg(reinterpret_cast<const uint4*>(src + 8));
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    c[i] = e4m3x2_from_f32(f.x * inv, f.y * inv);
  }
  return make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                    c[6] | (c[7] << 16));
}

template <int D>
__global__ void __launch_bounds__(256) reshape_and_cache_fp8_kernel(const CacheArgs a) {
  constexpr int kChunks = D / 16;  // 16-byte chunks (16 codes) per (token, head) row
  grid_launch_dependents();
  const int64_t total = a.num_tokens * a.num_kv_heads * kChunks;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ch = static_cast<int>(idx % kChunks);
    const int64_t row = idx / kChunks;
    const int h = static_cast<int>(row % a.num_kv_heads);
    const int64_t t = row / a.num_kv_heads;
    const int64_t slot = a.slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= a.num_blocks * a.block_size) {
      atomicOr(a.err, kErrSlotRange);
      continue;
    }
    const int64_t blk = slot / a.block_size;
    const int64_t off = slot % a.block_size;
    const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * D + ch * 16;
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.k_cache) + dst) =
        quantize16(a.k + t * a.k_stride + h * D + ch * 16, a.k_inv);
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.v_cache) + dst) =
        quantize16(a.v + t * a.v_stride + h * D + ch * 16, a.v_inv);
  }
}

// Copy-on-write of whole blocks: pair p (grid row y, strided) copies K and V of every kv head of
// block src to block dst with 16-byte loads and stores; grid columns split a block's chunks.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyArgs a) {
  for (int64_t p = blockIdx.y; p < a.num_pairs; p += gridDim.y) {
    const int32_t src = a.pairs[2 * p], dst = a.pairs[2 * p + 1];
    if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.err, kErrBlockRange);
      continue;
    }
    const int64_t s0 = src * a.chunks_per_block, d0 = dst * a.chunks_per_block;
    for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
         c < a.chunks_per_block; c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const uint4 k = a.k_cache[s0 + c], v = a.v_cache[s0 + c];
      a.k_cache[d0 + c] = k;
      a.v_cache[d0 + c] = v;
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream) {
  if (a.num_pairs == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t cols = (a.chunks_per_block + threads - 1) / threads;
  dim3 grid(static_cast<unsigned>(cols < 8 ? cols : 8),
            static_cast<unsigned>(a.num_pairs < 65535 ? a.num_pairs : 65535));
  copy_blocks_kernel<<<grid, threads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const CacheArgs& a, cudaStream_t stream) {
  const int64_t total = a.num_tokens * a.num_kv_heads * (a.head_dim / (a.fp8 ? 16 : 8));
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 152 * 64 ? want : 152 * 64);
  if (a.fp8) {
    if (a.head_dim == 128)
      reshape_and_cache_fp8_kernel<128><<<blocks, threads, 0, stream>>>(a);
    else
      reshape_and_cache_fp8_kernel<64><<<blocks, threads, 0, stream>>>(a);
  } else if (a.head_dim == 128) {
    reshape_and_cache_kernel<128><<<blocks, threads, 0, stream>>>(a);
  } else {
    reshape_and_cache_kernel<64><<<blocks, threads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pa
