// Decode attention over a paged KV cache: split-context partition kernel + log-sum-exp merge.
//
// Work item = one CTA = (sequence s, kv head g, partition p of 512 keys) for every sequence
// whose step has exactly one query row.  The CTA serves all G query heads of the GQA group
// from a single read of the group's K/V ("Local_LLM_03_vLLM_Architecture", KV-sizing slide:
// GQA-8; paged-KV slide: the kernel gathers K/V from scattered physical blocks).
//
// Data path per CTA (4 warps, each with a private ring of shared-memory stages):
//   * the partition's block ids are read from the block table once (block -> TMA row),
//   * each 16-token unit of K and of V (one or two 128-byte swizzled boxes per token row) is
//     fetched by a 2-D TMA tensor load that completes on the stage's mbarrier (its lines enter
//     L2 as the first to evict: they are read once); warp w takes units w, w+4, w+8, ... so one
//     partition keeps 4 x stages loads in flight per CTA,
//   * S^T = K Q^T on tensor cores (m16n8k16: 16 tokens x 8 heads x 16 dims), scores scaled by
//     scale*log2(e), masked past seq_len with a select (never arithmetic), online softmax
//     (running max / sum per head, exp2), P^T moved into the B-operand layout by movmatrix,
//     O^T += V^T P^T on tensor cores with V^T fed by ldmatrix.trans and the V rows past seq_len
//     (last unit only) zeroed in shared memory first (0 * NaN would poison the sum),
//   * the 4 warps' (m, l, O) are combined in shared memory; a single-partition sequence writes
//     fp16 output directly, otherwise the partition writes fp32 (m, l, O/l) partials that the
//     merge kernel combines:  M = max m_p,  w_p = 2^(m_p - M) l_p,  out = sum w_p o_p / sum w_p.
// FP8 (E4M3) cache: a unit is 16 rows of d bytes (one TMA box each for K and V, half the bytes).
// The MMA fragments are built from the codes directly (ldmatrix on the byte rows, then an exact
// E4M3 -> fp16 conversion in registers): a non-transposing ldmatrix gives a lane 4 consecutive
// codes of one token, which fill the A fragment of S^T = K Q^T under a permutation of the head
// dimension inside each 16-wide step (Q's B fragment uses the same one, so q.k is unchanged); a
// transposing ldmatrix gives 2 tokens x 2 dims, which fill the A fragment of V^T under a
// permutation of its rows (m-row i <-> dim 2i, m-row i + 8 <-> dim 2i + 1), undone when O is
// written out.  k_scale is folded into the score scale and v_scale multiplies the outputs.
// bfloat16 cache (with bf16 q and out): the fp16 data path with bf16 MMAs, P rounded to bf16
// for the P V product, and bf16 outputs.
// Both kernels are programmatic dependents of what precedes them on the stream: they may be
// scheduled early and read their descriptor and block table at once, but nothing that the
// kernel before them writes (the pools, the partials) before griddepcontrol.wait.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {
namespace {

template <int D, int BS, int NT, bool F8>
struct DecodeCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kHalves = D / 64;                // 128-byte fp16 boxes per token row
  static constexpr int kBoxBytes = 16 * 128;            // 16 token rows x 128 B
  static constexpr int kF16Bytes = kHalves * kBoxBytes; // fp16 K (or V) of one 16-token unit
  static constexpr int kKBytes = F8 ? 16 * D : kF16Bytes;  // K of one unit as stored in a stage
  static constexpr int kStageBytes = 2 * kKBytes;       // K + V
  // FP8: 3 stages of 4 KB per warp keep the bytes in flight per SM and fit 4 CTAs per SM.
  static constexpr int kStages = (F8 ? 48 * 1024 : 64 * 1024) / (kWarps * kStageBytes);
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
  static constexpr int kUnitsPerPart = kPartitionTokens / 16;
  static constexpr int kDK = D / 16;
  static constexpr int kHeads = NT * 8;
  static constexpr int kMergeBytes = kWarps * kHeads * (D + 2) * 4;
  static constexpr int kSmemBytes = (kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes) + 1024;
  // The running max is raised only past 2^8: p < 256 is exact enough in fp16 / bf16 (the same
  // relative rounding at every magnitude) and 512 keys of it stay far from fp32 overflow.
  static constexpr float kRaiseLog2 = 8.f;
  static_assert(kStages >= 1, "stage ring");
  static_assert(BS % 16 == 0, "block size must be a multiple of the 16-token unit");
};

// Shared-memory address of 16-byte chunk `chunk` of token row `tok` of an E4M3 unit as the TMA box
// lands: 128-byte swizzled rows for D = 128, plain 64-byte rows for D = 64.
template <int D>
__device__ __forceinline__ uint32_t f8_row_chunk(uint32_t base, int tok, int chunk) {
  return D == 128 ? base + tok * 128 + ((chunk ^ (tok & 7)) << 4) : base + tok * 64 + chunk * 16;
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

__device__ __forceinline__ uint32_t ldg_u32(const __half* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// What the pools hold: fp16, E4M3 codes (with fp16 q/out), or bf16 (with bf16 q/out).
enum KvKind : int { kKvF16 = 0, kKvE4M3 = 1, kKvBF16 = 2 };

// CAUSAL: the launch serves verify rows (several query rows per sequence), each column with its
// own causal limit; without it every column sees all L keys (decode rows only).
template <int D, int BS, int NT, int KV, bool CAUSAL>
__global__ void __launch_bounds__(DecodeCfg<D, BS, NT, KV == kKvE4M3>::kThreads, NT == 1 ? 4 : 0)
    decode_partition_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  constexpr bool F8 = KV == kKvE4M3, BF = KV == kKvBF16;
  using C = DecodeCfg<D, BS, NT, F8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[C::kWarps][C::kStages];
  __shared__ int32_t unit_row[C::kUnitsPerPart];

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // Grid x = (partition, column group), column group fastest so the CTAs that read the same
  // partition run side by side.  A column is one (query row, head of the group) pair, row-major;
  // a CTA serves 8 * NT of the sequence's q_len * G columns.  Partitions inside a shared prefix
  // belong to the shared-prefix pass and get no CTA here.
  const int ncg = a.col_groups;
  const int cg = static_cast<int>(blockIdx.x) % ncg;
  const int pidx = static_cast<int>(blockIdx.x) / ncg;
  const int part = pidx + a.cascade_parts, g = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = blockIdx.x == 0;  // reports the sequence's descriptor errors
  // The kernel before this one on the stream (the scatter-write) writes only the pools: the
  // descriptor and the block table are read before waiting for it, and only the K/V copies wait
  // (griddepcontrol.wait below), so the first wave's set-up overlaps that kernel.  q is read
  // after the first copies are issued, while they are in flight.
  grid_launch_dependents();
  // A CTA that leaves early still waits first, so that this grid never completes before the
  // one it depends on (the stream's order stays transitive for the launches after it).
  auto leave = [] { grid_dependency_wait(); };

  // One round of loads: the row range, the length, and the block ids of this partition's units
  // (thread u: unit u), read before the length is known: every column inside the table is a
  // valid address, and ids past the sequence's keys are never used.
  const int row0 = a.query_start_loc[s];
  const int row_end = a.query_start_loc[s + 1];
  const int L = a.seq_lens[s];
  int32_t unit_blk = 0;
  {
    const int col = (part * kPartitionTokens + tid * 16) / BS;
    if (tid < C::kUnitsPerPart && col < a.max_blocks)
      unit_blk = a.block_tables[static_cast<int64_t>(s) * a.bt_stride + col];
  }
  const int q_len = row_end - row0;
  // decode rows, and verify rows (a few per sequence) when the call routes them here
  if (q_len < 1 || q_len > a.verify_rows) return leave();
  if (row0 < 0 || row0 + q_len > a.num_tokens) {
    if (lead && tid == 0) atomicOr(a.err, kErrDescriptor);
    return leave();
  }
  const int nparts = (L + kPartitionTokens - 1) / kPartitionTokens;
  if (L < q_len || (L + BS - 1) / BS > a.max_blocks) {
    if (lead && tid == 0) atomicOr(a.err, kErrDescriptor);
    return leave();
  }
  if (nparts > static_cast<int>(gridDim.x) / ncg + a.cascade_parts ||
      (q_len * a.group + 8 * NT - 1) / (8 * NT) > ncg) {
    if (lead && tid == 0) atomicOr(a.err, kErrHint);
    return leave();
  }
  const int ncols = q_len * a.group, col0 = cg * 8 * NT;
  if (col0 >= ncols) return leave();
  const int ctx = L - q_len;  // row i sees keys 0 .. ctx + i
  if (a.cascade_parts > 0 && pidx == 0 && cg == 0 && g == 0) {
    // With a shared prefix, the row must have keys past it, and its table must hold sequence
    // 0's blocks inside it (the blocks the shared-prefix pass reads for every row).
    int differs = L <= a.cascade_parts * kPartitionTokens;
    const int nb = a.cascade_parts * (kPartitionTokens / BS);
    for (int j = tid; j < nb; j += C::kThreads)
      differs |= a.block_tables[static_cast<int64_t>(s) * a.bt_stride + j] != a.block_tables[j];
    if (__syncthreads_or(differs) && tid == 0) atomicOr(a.err, kErrDescriptor);
  }
  if (part >= nparts) return leave();

  const int tok_begin = part * kPartitionTokens;
  const int tok_end = min(L, tok_begin + kPartitionTokens);
  const int nunits = (tok_end - tok_begin + 15) >> 4;

  // Block id -> TMA row of every unit of the partition; ids outside the pool stop the CTA.
  static_assert(C::kUnitsPerPart <= C::kThreads, "one thread per unit");
  int bad = 0;
  if (tid < nunits) {
    const int tok = tok_begin + tid * 16;
    int y = 0;
    if (unit_blk >= 0 && unit_blk < a.num_blocks)
      y = (unit_blk * a.num_kv_heads + g) * BS + (tok % BS);
    else
      bad = 1;
    unit_row[tid] = y;
  }
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < C::kStages; ++st) mbar_init(smem_addr(&bars[warp][st]), 1);
    mbar_init_fence();
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(a.err, kErrBlockRange);
    return leave();
  }

  const int my_n = warp < nunits ? (nunits - warp + C::kWarps - 1) / C::kWarps : 0;
  const uint32_t ring = smem_addr(smem + warp * (C::kStages * C::kStageBytes));
  const uint32_t bar0 = smem_addr(&bars[warp][0]);

  // Every K/V line is read by this CTA alone, once: it goes into L2 as the first to evict, so
  // the stream does not push out what is read again (the partials the merge reads, the K/V
  // tiles a prefill grid beside this one shares among its CTAs, the block tables).
  const uint64_t pol = l2_policy_evict_first();
  auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y, uint32_t bar) {
    tma_load_2d_hint(dst, m, x, y, bar, pol);
  };
  auto issue = [&](int i) {  // lane 0: fetch unit i of this warp into stage i % kStages
    const int u = warp + i * C::kWarps;
    const int st = i % C::kStages;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t kdst = ring + st * C::kStageBytes;
    const int y = unit_row[u];
    mbar_arrive_expect_tx(bar, C::kStageBytes);
    if constexpr (F8) {  // one box of 16 rows x D bytes each
      load(kdst, &kmap, 0, y, bar);
      load(kdst + C::kKBytes, &vmap, 0, y, bar);
    } else {
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h) {
        load(kdst + h * C::kBoxBytes, &kmap, h * 64, y, bar);
        load(kdst + C::kKBytes + h * C::kBoxBytes, &vmap, h * 64, y, bar);
      }
    }
  };
  grid_dependency_wait();  // the pools now hold everything the previous kernels wrote
  if (lane == 0) {
    const int n0 = my_n < C::kStages ? my_n : C::kStages;
    for (int i = 0; i < n0; ++i) issue(i);
  }

  // Q^T as the B operand (k = head_dim, n = this CTA's columns), kept in registers.
  const int gq = lane >> 2, cq = lane & 3;
  uint32_t qf[NT][C::kDK][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int c = col0 + nt * 8 + gq;
    const bool hv = c < ncols;
    const int qi = hv ? c / a.group : 0, hg = hv ? c % a.group : 0;
    const __half* qrow = a.q + static_cast<int64_t>(row0 + qi) * a.q_stride +
                         static_cast<int64_t>(g * a.group + hg) * D;
#pragma unroll
    for (int j = 0; j < C::kDK; ++j) {
      // FP8: k positions (2cq, 2cq+1 | 2cq+8, 2cq+9) hold dims (4cq, 4cq+1 | 4cq+2, 4cq+3)
      qf[nt][j][0] = hv ? ldg_u32(qrow + j * 16 + (F8 ? 4 * cq : 2 * cq)) : 0u;
      qf[nt][j][1] = hv ? ldg_u32(qrow + j * 16 + (F8 ? 4 * cq + 2 : 8 + 2 * cq)) : 0u;
    }
  }

  // Last key position each of this lane's accumulator columns (2cq, 2cq + 1 of each 8) may see:
  // the causal limit of its query row (L - 1 for a decode row; columns past ncols see all).
  int lim[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int c = col0 + nt * 8 + 2 * cq + e;
      lim[nt][e] = c < ncols ? ctx + c / a.group : L - 1;
    }

  float o[NT][C::kDK][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int dt = 0; dt < C::kDK; ++dt) o[nt][dt][0] = o[nt][dt][1] = o[nt][dt][2] = o[nt][dt][3] = 0.f;
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }

  const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix index and row of this lane
  int failed_at = -1;
  for (int i = 0; i < my_n; ++i) {
    const int st = i % C::kStages;
    const bool ok = mbar_wait(bar0 + st * 8, (i / C::kStages) & 1, a.err, a.wait_limit_ns);
    if (__any_sync(0xffffffffu, !ok)) {
      failed_at = i;
      break;
    }
    const int u = warp + i * C::kWarps;
    const int nvalid = min(16, tok_end - (tok_begin + u * 16));
    const uint32_t kb = ring + st * C::kStageBytes;
    const uint32_t vb = kb + C::kKBytes;

    // ---- S^T[16 tokens][8 heads] = K Q^T
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    if constexpr (F8) {
      // one ldmatrix.x4 = two 16-dim steps x two 8-token halves of E4M3 codes
#pragma unroll
      for (int jj = 0; jj < C::kDK / 2; ++jj) {
        uint32_t r[4];
        ldsm_x4(f8_row_chunk<D>(kb, mr + ((mi & 1) << 3), 2 * jj + (mi >> 1)), r);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t af[4] = {f16x2_from_e4m3x2(r[2 * h]), f16x2_from_e4m3x2(r[2 * h + 1]),
                                  f16x2_from_e4m3x2(r[2 * h] >> 16),
                                  f16x2_from_e4m3x2(r[2 * h + 1] >> 16)};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816<BF>(sacc[nt], af, qf[nt][2 * jj + h][0], qf[nt][2 * jj + h][1]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < C::kDK; ++j) {
        const int tok = mr + ((mi & 1) << 3);
        const int chunk = 2 * j + (mi >> 1);
        uint32_t af[4];
        ldsm_x4(kb + (chunk >> 3) * C::kBoxBytes + swz128(tok, chunk & 7), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816<BF>(sacc[nt], af, qf[nt][j][0], qf[nt][j][1]);
      }
    }

    // ---- online softmax over the unit (per column; this lane holds columns 2cq, 2cq+1).
    // The running max m is a reference, not the exact max: it is raised (with the exact max of
    // the columns so far, rescaling l and O) only when some score of the warp passes it by more
    // than kRaiseLog2, so p = 2^(s - m) stays below 2^kRaiseLog2 and the usual unit needs no
    // cross-lane reduction and no rescale.  l and O are sums against the same m, so O / l is
    // the same quotient whatever m is.
    const int kp0 = tok_begin + u * 16 + gq, kp1 = kp0 + 8;  // key positions of rows gq, gq+8
    const bool v0 = gq < nvalid, v1 = gq + 8 < nvalid;
    float sc[NT][4];
    bool raise = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const bool c00 = !CAUSAL || kp0 <= lim[nt][0], c01 = !CAUSAL || kp0 <= lim[nt][1];
      const bool c10 = !CAUSAL || kp1 <= lim[nt][0], c11 = !CAUSAL || kp1 <= lim[nt][1];
      sc[nt][0] = v0 && c00 ? sacc[nt][0] * a.scale_log2 : -INFINITY;
      sc[nt][1] = v0 && c01 ? sacc[nt][1] * a.scale_log2 : -INFINITY;
      sc[nt][2] = v1 && c10 ? sacc[nt][2] * a.scale_log2 : -INFINITY;
      sc[nt][3] = v1 && c11 ? sacc[nt][3] * a.scale_log2 : -INFINITY;
      // m = -inf (no key seen yet) is passed by any visible score
      raise |= fmaxf(sc[nt][0], sc[nt][2]) > m_run[nt][0] + C::kRaiseLog2;
      raise |= fmaxf(sc[nt][1], sc[nt][3]) > m_run[nt][1] + C::kRaiseLog2;
    }
    if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float mx0 = fmaxf(sc[nt][0], sc[nt][2]), mx1 = fmaxf(sc[nt][1], sc[nt][3]);
        mx0 = warp_max_xor(mx0, 4);
        mx1 = warp_max_xor(mx1, 4);
        mx0 = warp_max_xor(mx0, 8);
        mx1 = warp_max_xor(mx1, 8);
        mx0 = warp_max_xor(mx0, 16);
        mx1 = warp_max_xor(mx1, 16);
        const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
        // a verify column with no visible key yet keeps m = -inf; its l and O are still 0
        const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m_run[nt][0] - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m_run[nt][1] - mn1);
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
        l_run[nt][0] *= al0;
        l_run[nt][1] *= al1;
#pragma unroll
        for (int dt = 0; dt < C::kDK; ++dt) {
          o[nt][dt][0] *= al0;
          o[nt][dt][1] *= al1;
          o[nt][dt][2] *= al0;
          o[nt][dt][3] *= al1;
        }
      }
    }
    uint32_t pb0[NT], pb1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // subtract 0 from a column still at m = -inf, so its (all -inf) scores give p = 0, not NaN
      const float b0 = CAUSAL && m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0];
      const float b1 = CAUSAL && m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1];
      const float p00 = exp2f(sc[nt][0] - b0), p10 = exp2f(sc[nt][2] - b0);
      const float p01 = exp2f(sc[nt][1] - b1), p11 = exp2f(sc[nt][3] - b1);
      l_run[nt][0] += p00 + p10;
      l_run[nt][1] += p01 + p11;
      pb0[nt] = movmatrix_trans(pack2<BF>(p00, p01));  // P^T[tok 2cq..2cq+1][head gq]
      pb1[nt] = movmatrix_trans(pack2<BF>(p10, p11));  // P^T[tok 2cq+8..][head gq]
    }

    // ---- O^T[d][heads] += V^T[d][16 tokens] P^T.  In a sequence's last, partial unit the V
    // rows past its end are zeroed in the stage first: their p is 0, but the rows may hold any
    // bits, and 0 * NaN would poison the sum.  (A whole token row is zeroed, so the swizzle of
    // its 16-byte chunks does not matter.)
    if (nvalid < 16) {
      constexpr int kRowChunks = F8 ? D / 16 : 2 * D / 16;  // 16-byte chunks per token row
      for (int c = lane; c < (16 - nvalid) * kRowChunks; c += 32) {
        const int row = nvalid + c / kRowChunks, k = c % kRowChunks;
        st_shared_zero16(F8 ? vb + row * D + k * 16
                            : vb + (k >> 3) * C::kBoxBytes + row * 128 + (k & 7) * 16);
      }
      __syncwarp();
    }
    if constexpr (F8) {
      // one ldmatrix.x4.trans = two 16-dim blocks x two 8-token halves; a lane holds, per
      // matrix, tokens (2cq, 2cq+1) x dims (2gq, 2gq+1) of the block: bytes 0, 2 are dim 2gq
      // (m-row gq), bytes 1, 3 dim 2gq + 1 (m-row gq + 8)
#pragma unroll
      for (int dd = 0; dd < C::kDK / 2; ++dd) {
        uint32_t r[4];
        ldsm_x4_trans(f8_row_chunk<D>(vb, mr + ((mi & 1) << 3), 2 * dd + (mi >> 1)), r);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t af[4] = {f16x2_from_e4m3x2(__byte_perm(r[2 * h], 0, 0x3320)),
                                  f16x2_from_e4m3x2(__byte_perm(r[2 * h], 0, 0x3331)),
                                  f16x2_from_e4m3x2(__byte_perm(r[2 * h + 1], 0, 0x3320)),
                                  f16x2_from_e4m3x2(__byte_perm(r[2 * h + 1], 0, 0x3331))};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816<BF>(o[nt][2 * dd + h], af, pb0[nt], pb1[nt]);
        }
      }
    } else {
#pragma unroll
      for (int dt = 0; dt < C::kDK; ++dt) {
        const int tok = mr + ((mi >> 1) << 3);
        const int chunk = 2 * dt + (mi & 1);
        uint32_t af[4];
        ldsm_x4_trans(vb + (chunk >> 3) * C::kBoxBytes + swz128(tok, chunk & 7), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816<BF>(o[nt][dt], af, pb0[nt], pb1[nt]);
      }
    }

    __syncwarp();
    if (lane == 0 && i + C::kStages < my_n) {
      fence_proxy_async();
      issue(i + C::kStages);
    }
  }

  if (failed_at >= 0) {
    // A copy never arrived: let whatever is still in flight land (bounded) before leaving.
    if (lane == 0) {
      const int issued = min(my_n, failed_at + C::kStages);
      for (int i = failed_at + 1; i < issued; ++i)
        mbar_wait(bar0 + (i % C::kStages) * 8, (i / C::kStages) & 1, a.err, a.wait_limit_ns);
    }
  }

  // ---- combine the warps' partial softmax states
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[nt][e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      l_run[nt][e] = l;
    }
  }
  __syncthreads();  // every warp is done with its ring: reuse it for the merge
  constexpr int H = C::kHeads;
  float* sm_m = reinterpret_cast<float*>(smem);
  float* sm_l = sm_m + C::kWarps * H;
  float* sm_o = sm_l + C::kWarps * H;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = nt * 8 + 2 * cq + e;
      if (gq == 0) {
        sm_m[warp * H + h] = m_run[nt][e];
        sm_l[warp * H + h] = l_run[nt][e];
      }
      float* dst = sm_o + (warp * H + h) * D;
#pragma unroll
      for (int dt = 0; dt < C::kDK; ++dt) {
        // m-rows gq, gq + 8 of O^T: dims gq, gq + 8 (fp16) or 2gq, 2gq + 1 (FP8 permutation)
        dst[dt * 16 + (F8 ? 2 * gq : gq)] = o[nt][dt][e];
        dst[dt * 16 + (F8 ? 2 * gq + 1 : gq + 8)] = o[nt][dt][2 + e];
      }
    }
  }
  // A warp that timed out has set the error word; the whole CTA then leaves its outputs alone.
  if (__syncthreads_or(failed_at >= 0)) return;

  const int my_cols = min(8 * NT, ncols - col0);
  for (int idx = tid; idx < my_cols * D; idx += C::kThreads) {
    const int h = idx / D, d = idx % D;  // h: the CTA's column
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, sm_m[w * H + h]);
    const float base = M == -INFINITY ? 0.f : M;  // the row sees no key of this partition
    float wsum = 0.f, osum = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float f = exp2f(sm_m[w * H + h] - base);
      wsum += f * sm_l[w * H + h];
      osum += f * sm_o[(w * H + h) * D + d];
    }
    const int c = col0 + h;
    const int hq = g * a.group + c % a.group;
    const int64_t orow = static_cast<int64_t>(row0 + c / a.group) * a.num_q_heads + hq;
    if (nparts == 1) {
      store_elem<BF>(a.out + orow * D + d, osum / wsum * a.v_scale);
    } else {
      const int64_t pi = orow * a.max_parts + part;
      a.part_o[pi * D + d] = wsum > 0.f ? osum / wsum * a.v_scale : 0.f;
      if (d == 0) {
        a.part_m[pi] = M;
        a.part_l[pi] = wsum;
      }
    }
  }
}

// One warp per (query row, head) of the rows the decode kernel served (grid z = row of the
// sequence): combine the row's partitions.  Two dependent memory rounds: the row's descriptor
// (query_start_loc and seq_lens together), then every partition's m and l with the first 16
// partitions' O rows, all in flight at once.  A partition past a verify row's causal limit
// holds l = 0, O = 0 and weighs nothing.
template <int D, bool BF>
__global__ void __launch_bounds__(128) merge_partitions_kernel(const AttnArgs a) {
  grid_launch_dependents();
  auto leave = [] { grid_dependency_wait(); };  // as in the decode kernel
  const int s = blockIdx.y, qi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.x * 4 + warp;
  if (hq >= a.num_q_heads) return leave();
  const int row0 = a.query_start_loc[s], row1 = a.query_start_loc[s + 1];
  const int L = a.seq_lens[s];
  const int q_len = row1 - row0;
  if (q_len < 1 || q_len > a.verify_rows || qi >= q_len || row0 < 0 || row1 > a.num_tokens ||
      L < q_len)
    return leave();
  const int nparts = (L + kPartitionTokens - 1) / kPartitionTokens;
  if (nparts <= 1 || nparts > a.max_parts || (L + a.block_size - 1) / a.block_size > a.max_blocks)
    return leave();
  const int row = row0 + qi;
  const int64_t base = (static_cast<int64_t>(row) * a.num_q_heads + hq) * a.max_parts;
  grid_dependency_wait();  // the partials come from the kernels before (descriptor: an input)

  constexpr int V = D / 32;   // output elements per lane
  constexpr int kBatch = 16;  // partitions whose O rows are in flight at once
  constexpr int kHeld = 2;    // m and l of partitions lane, lane + 32 held in registers
  // A shared-prefix CTA that covered several prefix partitions wrote its partial to the first
  // one's slot; the others hold nothing and weigh nothing.
  auto unused = [&](int p) { return p < a.cascade_parts && p % a.cascade_span != 0; };
  auto load_o = [&](int p, float (&x)[V]) {
    if (unused(p)) {
#pragma unroll
      for (int e = 0; e < V; ++e) x[e] = 0.f;
      return;
    }
    const float* op = a.part_o + (base + p) * D + lane * V;
    if constexpr (V == 4) {
      const float4 t = *reinterpret_cast<const float4*>(op);
      x[0] = t.x, x[1] = t.y, x[2] = t.z, x[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(op);
      x[0] = t.x, x[1] = t.y;
    }
  };
  float mh[kHeld], lh[kHeld];
#pragma unroll
  for (int k = 0; k < kHeld; ++k) {
    const int p = lane + 32 * k;
    mh[k] = p < nparts && !unused(p) ? a.part_m[base + p] : -INFINITY;
    lh[k] = p < nparts && !unused(p) ? a.part_l[base + p] : 0.f;
  }
  float x[kBatch][V];
#pragma unroll
  for (int j = 0; j < kBatch; ++j)
    if (j < nparts) load_o(j, x[j]);
  float M = -INFINITY;
  for (int p = lane + 32 * kHeld; p < nparts; p += 32)
    if (!unused(p)) M = fmaxf(M, a.part_m[base + p]);
#pragma unroll
  for (int k = 0; k < kHeld; ++k) M = fmaxf(M, mh[k]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  // weight of partition p: 2^(m_p - M) l_p, held by lane p % 32 in register p / 32
  float wh[kHeld];
#pragma unroll
  for (int k = 0; k < kHeld; ++k) wh[k] = exp2f(mh[k] - M) * lh[k];

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int p0 = 0; p0 < nparts; p0 += kBatch) {
    const int n = min(kBatch, nparts - p0);
    if (p0 > 0) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (j < n) load_o(p0 + j, x[j]);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int p = p0 + j;  // the same for every lane
      if (j < n) {
        float wj;
        if (p < 32 * kHeld) {
          float src = wh[0];
#pragma unroll
          for (int k = 1; k < kHeld; ++k) src = (p >> 5) == k ? wh[k] : src;
          wj = __shfl_sync(0xffffffffu, src, p & 31);
        } else {  // past 32 * kHeld partitions: read m and l again (the same address in every lane)
          wj = unused(p) ? 0.f : exp2f(a.part_m[base + p] - M) * a.part_l[base + p];
        }
        wsum += wj;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] += wj * x[j][e];
      }
    }
  }
  __half* dst = a.out + (static_cast<int64_t>(row) * a.num_q_heads + hq) * D + lane * V;
  const float inv = 1.f / wsum;
  if constexpr (V == 4) {
    uint2 pk;
    pk.x = pack2<BF>(acc[0] * inv, acc[1] * inv);
    pk.y = pack2<BF>(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack2<BF>(acc[0] * inv, acc[1] * inv);
  }
}

template <int D, int BS, int NT, int KV, bool CAUSAL>
cudaError_t launch_decode_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  using C = DecodeCfg<D, BS, NT, KV == kKvE4M3>;
  auto kern = decode_partition_kernel<D, BS, NT, KV, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.max_parts - a.cascade_parts) * a.col_groups, a.num_kv_heads, a.num_seqs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a);
}

template <int D, int BS, int KV>
cudaError_t launch_decode_g(const AttnArgs& a, const CUtensorMap& k, const CUtensorMap& v,
                            cudaStream_t st) {
  // 8 columns per CTA while the widest sequence's q_len x G fits, else 16 per CTA
  if (a.verify_rows > 1)
    return a.group * a.verify_rows <= 8 ? launch_decode_t<D, BS, 1, KV, true>(a, k, v, st)
                                        : launch_decode_t<D, BS, 2, KV, true>(a, k, v, st);
  return a.group <= 8 ? launch_decode_t<D, BS, 1, KV, false>(a, k, v, st)
                      : launch_decode_t<D, BS, 2, KV, false>(a, k, v, st);
}

template <int D, int BS>
cudaError_t launch_decode_f(const AttnArgs& a, const CUtensorMap& k, const CUtensorMap& v,
                            cudaStream_t st) {
  if (a.kv_fp8) return launch_decode_g<D, BS, kKvE4M3>(a, k, v, st);
  return a.bf16 ? launch_decode_g<D, BS, kKvBF16>(a, k, v, st)
                : launch_decode_g<D, BS, kKvF16>(a, k, v, st);
}

}  // namespace

cudaError_t launch_decode(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.block_size == 16 ? launch_decode_f<128, 16>(a, kmap, vmap, stream)
                              : launch_decode_f<128, 32>(a, kmap, vmap, stream);
  return a.block_size == 16 ? launch_decode_f<64, 16>(a, kmap, vmap, stream)
                            : launch_decode_f<64, 32>(a, kmap, vmap, stream);
}

cudaError_t launch_merge(const AttnArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.num_q_heads + 3) / 4, a.num_seqs, a.verify_rows);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.bf16)
    return a.head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_partitions_kernel<128, true>, a)
                             : cudaLaunchKernelEx(&cfg, merge_partitions_kernel<64, true>, a);
  return a.head_dim == 128 ? cudaLaunchKernelEx(&cfg, merge_partitions_kernel<128, false>, a)
                           : cudaLaunchKernelEx(&cfg, merge_partitions_kernel<64, false>, a);
}

}  // namespace pa
