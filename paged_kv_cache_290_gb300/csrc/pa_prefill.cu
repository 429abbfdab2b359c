// Chunked-prefill attention over a paged KV cache.
//
// A prefill chunk of q_len rows for a sequence of seq_len keys sits at absolute positions
// ctx .. ctx + q_len - 1 with ctx = seq_len - q_len; row i attends to keys 0 .. ctx + i
// ("Local_LLM_03_vLLM_Architecture", chunked-prefill slide: a long prefill is cut into chunks,
// e.g. 512 tokens, interleaved with decodes; the chunk sees the paged context written before).
//
// Work item = one CTA = (q tile, sequence s, kv head g).  The tile's 128 rows are
// (query token, head of the GQA group) pairs, so one K/V tile in shared memory serves every
// head of the group.  A producer warp streams 64-key K and V tiles (four 16-token units,
// each one or two 128-byte-swizzled TMA boxes, gathered through the block table) into a
// two-stage ring; eight consumer warps each own 16 rows and run S = Q K^T and O += P V on
// tensor cores (m16n8k16, fp16 in, fp32 accumulate) with an online softmax in exp2.
#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {
namespace {

template <int D, int BS>
struct PrefillCfg {
  static constexpr int kConsumers = 8;
  static constexpr int kThreads = (kConsumers + 1) * 32;
  static constexpr int kRows = kConsumers * 16;
  static constexpr int kKeys = 64;
  static constexpr int kUnits = kKeys / 16;
  static constexpr int kHalves = D / 64;
  static constexpr int kBoxBytes = 16 * 128;
  static constexpr int kUnitBytes = kHalves * kBoxBytes;
  static constexpr int kTileBytes = kUnits * kUnitBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = 2;
  static constexpr int kDK = D / 16;
  static constexpr int kDN = D / 8;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static_assert(BS % 16 == 0, "block size must be a multiple of the 16-token unit");
};

__device__ __forceinline__ uint32_t ldg_u32(const __half* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

template <int D, int BS>
__global__ void __launch_bounds__(PrefillCfg<D, BS>::kThreads, 1)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = PrefillCfg<D, BS>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int qt = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int row0 = a.query_start_loc[s];
  const int q_len = a.query_start_loc[s + 1] - row0;
  if (q_len <= 1) return;  // decode rows and idle sequences are handled elsewhere
  const int L = a.seq_lens[s];
  const int tile_q = C::kRows / a.group;  // query tokens per CTA
  const int qbase = qt * tile_q;
  if (q_len > L || (L + BS - 1) / BS > a.max_blocks || row0 < 0 ||
      row0 + q_len > a.num_tokens) {
    if (qt == 0 && tid == 0) atomicOr(a.err, kErrDescriptor);
    return;
  }
  if ((q_len + tile_q - 1) / tile_q > static_cast<int>(gridDim.x)) {
    if (qt == 0 && tid == 0) atomicOr(a.err, kErrHint);
    return;
  }
  if (qbase >= q_len) return;
  const int ctx = L - q_len;
  const int q_hi = min(q_len, qbase + tile_q);  // rows [qbase, q_hi) of the chunk
  const int kend = ctx + q_hi;                  // keys [0, kend) are visible to some row
  const int ntiles = (kend + C::kKeys - 1) / C::kKeys;

  // Validate every block id the CTA will read before any copy is issued.
  int bad = 0;
  const int nblk = (kend + BS - 1) / BS;
  for (int j = tid; j < nblk; j += C::kThreads) {
    const int32_t blk = a.block_tables[static_cast<int64_t>(s) * a.bt_stride + j];
    if (blk < 0 || blk >= a.num_blocks) bad = 1;
  }
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(smem_addr(&full_bar[st]), 1);
      mbar_init(smem_addr(&empty_bar[st]), C::kConsumers);
    }
    mbar_init_fence();
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(a.err, kErrBlockRange);
    return;
  }
  const uint32_t ring = smem_addr(smem);

  if (warp == C::kConsumers) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % C::kStages;
        if (i >= C::kStages && !mbar_wait(smem_addr(&empty_bar[st]), ((i / C::kStages) - 1) & 1, a.err))
          break;
        const int key0 = i * C::kKeys;
        const int units = min(C::kUnits, (kend - key0 + 15) >> 4);
        const uint32_t bar = smem_addr(&full_bar[st]);
        mbar_arrive_expect_tx(bar, units * 2 * C::kUnitBytes);
        const uint32_t kdst = ring + st * C::kStageBytes;
        for (int u = 0; u < units; ++u) {
          const int tok = key0 + u * 16;
          const int32_t blk = a.block_tables[static_cast<int64_t>(s) * a.bt_stride + tok / BS];
          const int y = (blk * a.num_kv_heads + g) * BS + (tok % BS);
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_2d(kdst + u * C::kUnitBytes + h * C::kBoxBytes, &kmap, h * 64, y, bar);
            tma_load_2d(kdst + C::kTileBytes + u * C::kUnitBytes + h * C::kBoxBytes, &vmap,
                        h * 64, y, bar);
          }
        }
        issued = i + 1;
      }
      // Let the last copies land before the CTA can retire (bounded).
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(smem_addr(&full_bar[i % C::kStages]), (i / C::kStages) & 1, a.err);
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  const int gq = lane >> 2, cq = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;
  // Rows owned by this lane: R0 = warp*16 + gq and R1 = R0 + 8 -> (query token, head).
  int qi[2], hg[2], pos[2];
  bool rv[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int R = warp * 16 + gq + 8 * e;
    qi[e] = R / a.group;
    hg[e] = R % a.group;
    rv[e] = qi[e] < tile_q && qbase + qi[e] < q_len;
    pos[e] = ctx + (rv[e] ? qbase + qi[e] : qbase);  // padding rows mirror the first row
  }
  // Q as the A operand (row-major 16 x 16 per k step), kept in registers.
  uint32_t qa[C::kDK][4];
  {
    const __half* qp[2];
#pragma unroll
    for (int e = 0; e < 2; ++e)
      qp[e] = a.q + static_cast<int64_t>(row0 + qbase + (rv[e] ? qi[e] : 0)) * a.q_stride +
              static_cast<int64_t>(g * a.group + hg[e]) * D;
#pragma unroll
    for (int j = 0; j < C::kDK; ++j) {
      qa[j][0] = rv[0] ? ldg_u32(qp[0] + j * 16 + 2 * cq) : 0u;
      qa[j][1] = rv[1] ? ldg_u32(qp[1] + j * 16 + 2 * cq) : 0u;
      qa[j][2] = rv[0] ? ldg_u32(qp[0] + j * 16 + 8 + 2 * cq) : 0u;
      qa[j][3] = rv[1] ? ldg_u32(qp[1] + j * 16 + 8 + 2 * cq) : 0u;
    }
  }

  float o[C::kDN][4];
#pragma unroll
  for (int dn = 0; dn < C::kDN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int min_pos = ctx + qbase;  // keys up to here are visible to every row of the tile
  bool failed = false;

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::kStages;
    const bool ok = mbar_wait(smem_addr(&full_bar[st]), (i / C::kStages) & 1, a.err);
    if (__any_sync(0xffffffffu, !ok)) {
      failed = true;
      break;
    }
    const uint32_t kb = ring + st * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;
    const int key0 = i * C::kKeys;

    // ---- S[16 rows][64 keys] = Q K^T
    float sacc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int j = 0; j < C::kDK; ++j) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int row = mr + ((mi >> 1) << 3);  // key within the 16-key unit np
        const int chunk = 2 * j + (mi & 1);
        uint32_t bf[4];
        ldsm_x4(kb + np * C::kUnitBytes + (chunk >> 3) * C::kBoxBytes + swz128(row, chunk & 7), bf);
        mma_f16_16816(sacc[2 * np], qa[j], bf[0], bf[1]);
        mma_f16_16816(sacc[2 * np + 1], qa[j], bf[2], bf[3]);
      }
    }

    // ---- causal mask + online softmax (rows gq and gq+8 of this warp)
    const bool need_mask = key0 + C::kKeys - 1 > min_pos;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = c >> 1;
        const int key = key0 + nt * 8 + 2 * cq + (c & 1);
        float v = sacc[nt][c] * a.scale_log2;
        if (need_mask) v = key <= pos[e] ? v : -INFINITY;
        sacc[nt][c] = v;
        mx[e] = fmaxf(mx[e], v);
      }
    }
    float al[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = warp_max_xor(mx[e], 1);
      mx[e] = warp_max_xor(mx[e], 2);
      const float mn = fmaxf(m_run[e], mx[e]);
      al[e] = exp2f(m_run[e] - mn);
      m_run[e] = mn;
    }
    float ls[2] = {0.f, 0.f};
    uint32_t pa[4][4];  // P as the A operand for the 4 k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f(sacc[nt][0] - m_run[0]);
      const float p1 = exp2f(sacc[nt][1] - m_run[0]);
      const float p2 = exp2f(sacc[nt][2] - m_run[1]);
      const float p3 = exp2f(sacc[nt][3] - m_run[1]);
      ls[0] += p0 + p1;
      ls[1] += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_half2(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_half2(p2, p3);
    }
    l_run[0] = l_run[0] * al[0] + ls[0];
    l_run[1] = l_run[1] * al[1] + ls[1];
#pragma unroll
    for (int dn = 0; dn < C::kDN; ++dn) {
      o[dn][0] *= al[0];
      o[dn][1] *= al[0];
      o[dn][2] *= al[1];
      o[dn][3] *= al[1];
    }

    // ---- O[16 rows][d] += P V ; V rows at or past kend are zeroed (they may hold NaN)
    const bool tail = key0 + C::kKeys > kend;
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t m_lo = 0xffffffffu, m_hi = 0xffffffffu;
      if (tail) {
        const int k_lo = key0 + kt * 16 + 2 * cq, k_hi = k_lo + 8;
        m_lo = (k_lo < kend ? 0x0000ffffu : 0u) | (k_lo + 1 < kend ? 0xffff0000u : 0u);
        m_hi = (k_hi < kend ? 0x0000ffffu : 0u) | (k_hi + 1 < kend ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int dp = 0; dp < C::kDK; ++dp) {
        const int row = mr + ((mi & 1) << 3);
        const int chunk = 2 * dp + (mi >> 1);
        uint32_t bf[4];
        ldsm_x4_trans(vb + kt * C::kUnitBytes + (chunk >> 3) * C::kBoxBytes + swz128(row, chunk & 7), bf);
        bf[0] &= m_lo;
        bf[1] &= m_hi;
        bf[2] &= m_lo;
        bf[3] &= m_hi;
        mma_f16_16816(o[2 * dp], pa[kt], bf[0], bf[1]);
        mma_f16_16816(o[2 * dp + 1], pa[kt], bf[2], bf[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[st]));
  }
  if (failed) return;

#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 1);
    l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 2);
  }
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    if (!rv[e]) continue;
    const float inv = 1.f / l_run[e];
    __half* dst = a.out + (static_cast<int64_t>(row0 + qbase + qi[e]) * a.num_q_heads +
                           g * a.group + hg[e]) * D;
#pragma unroll
    for (int dn = 0; dn < C::kDN; ++dn)
      *reinterpret_cast<uint32_t*>(dst + dn * 8 + 2 * cq) =
          pack_half2(o[dn][2 * e] * inv, o[dn][2 * e + 1] * inv);
  }
}

template <int D, int BS>
cudaError_t launch_prefill_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  using C = PrefillCfg<D, BS>;
  auto kern = prefill_chunk_kernel<D, BS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int tile_q = C::kRows / a.group;
  dim3 grid((a.max_query_len + tile_q - 1) / tile_q, a.num_kv_heads, a.num_seqs);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.block_size == 16 ? launch_prefill_t<128, 16>(a, kmap, vmap, stream)
                              : launch_prefill_t<128, 32>(a, kmap, vmap, stream);
  return a.block_size == 16 ? launch_prefill_t<64, 16>(a, kmap, vmap, stream)
                            : launch_prefill_t<64, 32>(a, kmap, vmap, stream);
}

}  // namespace pa
