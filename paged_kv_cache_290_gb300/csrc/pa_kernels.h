// Host-side launch interface between the C ABI (pa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace pa {

struct CacheArgs {
  const __half* k;
  const __half* v;
  int64_t k_stride;  // elements between consecutive tokens of k
  int64_t v_stride;
  void* k_cache;  // fp16, or E4M3 bytes when fp8
  void* v_cache;
  int fp8;        // 1: store E4M3 codes of x * k_inv (v_inv)
  float k_inv;    // 1 / k_scale in float32
  float v_inv;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int64_t num_blocks;
  unsigned* err;
};

struct AttnArgs {
  const __half* q;
  int64_t q_stride;  // elements between consecutive query tokens
  __half* out;       // [T, Hq, d] contiguous
  const int32_t* block_tables;
  int64_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  float* part_o;  // [T, Hq, P, d]
  float* part_m;  // [T, Hq, P]
  float* part_l;  // [T, Hq, P]
  int num_seqs;
  int64_t num_tokens;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int head_dim;
  int block_size;
  int max_blocks;  // columns of block_tables
  int64_t num_blocks;
  int max_parts;   // P = ceil(max_seq_len / 512) (>= 1)
  int max_query_len;
  int prefill_seqs;  // sequences the prefill launch covers (<= num_seqs)
  int decode_skipped;  // 1: the hint promised no one-row sequence, so no decode launch was made
  float scale_log2;  // scale * log2(e) (times k_scale for an FP8 cache)
  float v_scale;     // FP8 cache: multiplies the output; 1 for fp16
  int kv_fp8;        // 1: the pools hold E4M3 codes
  int bf16;          // 1: q, out and the pools are bfloat16 (else fp16)
  int cascade_parts; // leading 512-key partitions every sequence shares (attended once for all)
  int cascade_span;  // prefix partitions one shared-prefix CTA covers (their partial goes to the
                     //   first one's slot; the merge skips the others)
  int num_sms;       // SMs of the device (launch-shape choices)
  int verify_rows;   // the decode kernel and its merge serve sequences with 1 .. verify_rows
                     //   query rows (1: decode rows only)
  int col_groups;    // decode CTAs per (sequence, kv head, partition): ceil(rows x G / columns)
  int items_x;       // > 0: the two-tile prefill kernel runs as launches over slices of its
                     //   items (x q-tile pairs per (kv head, sequence)); 0: one full grid
  int item_base;     // first item of such a launch
  int prefill_ctas;  // CTAs per such launch (0: one full grid)
  uint64_t wait_limit_ns;  // every bounded wait of the call gives up after this long
  unsigned* err;
};

// Sets the message pa_last_error() returns on this host thread; returns `status`.
int set_last_error(int status, const std::string& message);

// Device address of the error word a call on `stream` reports into: the word the caller
// registered for that stream, else the current device's (looked up once per device).
cudaError_t error_word(void* stream, unsigned** out);

// Whole-block copies (copy-on-write of shared blocks).
struct CopyArgs {
  uint4* k_cache;  // the pool as 16-byte chunks
  uint4* v_cache;
  const int32_t* pairs;  // [n][2] = (src, dst)
  int64_t num_pairs;
  int64_t chunks_per_block;  // Hkv * bs * d / 8
  int64_t num_blocks;
  unsigned* err;
};

cudaError_t launch_reshape_and_cache(const CacheArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream);
cudaError_t launch_merge(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream);
cudaError_t launch_shared_prefix(const AttnArgs& a, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pa
