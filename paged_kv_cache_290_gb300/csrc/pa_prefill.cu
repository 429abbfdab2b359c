// Chunked-prefill attention over a paged KV cache on the 5th-generation tensor cores.
//
// A prefill chunk of q_len rows for a sequence of seq_len keys sits at absolute positions
// ctx .. ctx + q_len - 1 with ctx = seq_len - q_len; row i attends to keys 0 .. ctx + i
// ("Local_LLM_03_vLLM_Architecture", chunked-prefill slide: a long prefill is cut into chunks,
// e.g. 512 tokens, interleaved with decodes; the chunk sees the paged context written before).
//
// Two kernels, chosen per launch by the longest chunk (the hint's max_query_len):
//   * prefill_pair_kernel when a chunk spans more than one 128-row Q tile, described below;
//   * prefill_parity_kernel when every chunk fits one Q tile (speculative verify, short chunks):
//     the same warp roles and TMEM layout, but its two softmax warpgroups take the even and the
//     odd key tiles of the one Q tile, each with its own online softmax and O accumulator, merged
//     at the end with the log-sum-exp rule (S_{j+2} reuses S_j's buffer after P_j V_j).
// Both find their sequence with a scan of the descriptor (the pair kernel in batch order, the
// parity kernel longest sequence first) and feed K/V with the same producer warps.
//
// prefill_pair_kernel: work item = one CTA = (two Q tiles, kv head g, prefill sequence).  A Q
// tile is 128 rows, each a (query token, head of the GQA group) pair, so one K/V tile serves
// every head of the group, and every K/V tile the CTA loads serves both Q tiles (256 rows).
// 640 threads; warp roles:
//   * producers (warps 16 and 17): stream 128-key K and V tiles (8 units of 16 tokens gathered
//     through the block table, 128-byte-swizzled TMA boxes) into a 2-stage K ring and a 3-stage
//     V ring; a K stage is released once both S = Q K^T products that read it are done, a V
//     stage as soon as both P V products are (before the next S is issued).  The next tile's
//     block ids are read while a producer waits for its stage, and the MMA issuer waits for
//     K_{j+1} only right before S(j+1),
//   * MMA issuer (lane 0 of warp 18): per Q tile t, S_t = Q_t K_j^T into TMEM buffer t (M 128,
//     N 128, K d, both operands K-major from shared memory) and O_t += P_t V_j with P_t read
//     from TMEM (it overwrites the first 64 columns of S_t's buffer, two fp16 per column) and
//     V_j MN-major from shared memory.  Issue order S_A(0), S_B(0), then per key tile j:
//     P_A V_j, S_A(j+1), P_B V_j, S_B(j+1): the tensor pipe computes one Q tile's products
//     while the other tile is in softmax, and since tcgen05 MMAs of one thread run in issue
//     order, S_t(j+1) never overwrites P_t(j) before P_t V_j has read it.  Issuing an MMA
//     waits until the pipe takes it, so this thread runs alone and never joins a warp
//     collective (that would idle the pipe),
//   * softmax (warps 0 .. 15): two warpgroups per Q tile t (warps 8t .. 8t+7), one per half of
//     each key tile's columns and of O's columns, a thread per (row, half); the two halves of a
//     row trade their maxima once per key tile through a named barrier.  Online softmax in base
//     2 with scale * log2(e) folded into the exponent, on packed fp32 pairs.  The running max is
//     only raised (and O_t rescaled in TMEM) when it grows by more than 8 in log2 units, which
//     keeps P <= 256 in fp16.  S_t(j)'s completion implies P_t V_{j-1} is done (it was issued
//     after it), so no softmax step waits on a P V,
//   * warp 19 widens half of each tile's E4M3 codes over an FP8 pool (d 128), else idles.
// V rows past the last visible key of the chunk are zeroed in shared memory before the first
// P V product of the last key tile (0 * NaN would poison the sum).  Every wait is bounded.
// A bfloat16 batch (q, pools and out bf16) runs the same kernels with bf16 operands in both
// products (kind::f16 takes A and B both fp16 or both bf16), P packed as bf16 into TMEM.
#include <algorithm>

#include "pa_common.cuh"
#include "pa_kernels.h"

namespace pa {
namespace {

// Grid row z of a prefill launch serves the z-th sequence with more than one query row (a
// block-wide ballot scan of query_start_loc, all threads of the CTA), so decode rows cost the
// launch nothing.  Returns that sequence, or -1 past the last one; more such sequences than
// grid rows (or, when the decode launch was skipped on the hint's word, a one-row sequence) is
// a hint error.
template <int kThreads>
__device__ __forceinline__ int find_prefill_seq(const AttnArgs& a, int* warp_count,
                                                int* chosen_seq, int target, bool first) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) *chosen_seq = -1;
  int found = 0;  // prefill sequences seen so far
  for (int s0 = 0; s0 < a.num_seqs; s0 += kThreads) {
    const int si = s0 + tid;
    const int ql = si < a.num_seqs ? a.query_start_loc[si + 1] - a.query_start_loc[si] : 0;
    const bool pf = ql > 1;
    const unsigned bal = __ballot_sync(0xffffffffu, pf);
    if (a.decode_skipped && __any_sync(0xffffffffu, ql == 1) && lane == 0 && first)
      atomicOr(a.err, kErrHint);
    if (lane == 0) warp_count[warp] = __popc(bal);
    __syncthreads();
    int rank = found + __popc(bal & ((1u << lane) - 1u)), total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      rank += w < warp ? warp_count[w] : 0;
      total += warp_count[w];
    }
    if (pf && rank == target) *chosen_seq = si;
    found += total;
    __syncthreads();
  }
  __syncthreads();
  if (found > a.prefill_seqs && first && tid == 0) atomicOr(a.err, kErrHint);
  return *chosen_seq;
}

// As find_prefill_seq, but grid row z serves the prefill sequence of rank z when they are
// ordered longest first (ties: batch order), so the longest CTAs are dispatched first and the
// grid's tail is short.  For the one-Q-tile kernel, whose CTAs share no K/V tile, so the order
// costs no L2 reuse.  The ranks are taken in one pass over at most kThreads sequences, through
// `scratch` (kThreads ints of dynamic shared memory that nothing uses yet); a larger batch keeps
// batch order.
template <int kThreads>
__device__ __forceinline__ int find_prefill_seq_longest_first(const AttnArgs& a, int* warp_count,
                                                              int* chosen_seq, int* scratch,
                                                              int target, bool first) {
  if (a.num_seqs > kThreads) return find_prefill_seq<kThreads>(a, warp_count, chosen_seq, target, first);
  const int tid = threadIdx.x;
  if (tid == 0) *chosen_seq = -1;
  const int ql = tid < a.num_seqs ? a.query_start_loc[tid + 1] - a.query_start_loc[tid] : 0;
  const bool pf = ql > 1;
  const int key = pf ? max(a.seq_lens[tid], 0) : -1;  // -1: not a prefill sequence
  if (first && a.decode_skipped && ql == 1) atomicOr(a.err, kErrHint);
  scratch[tid] = key;
  __syncthreads();
  int rank = 0, found = 0;
  for (int j = 0; j < a.num_seqs; ++j) {  // every thread reads the same word: a broadcast
    const int kj = scratch[j];
    found += kj >= 0;
    rank += kj > key || (kj == key && j < tid);
  }
  if (pf && rank == target) *chosen_seq = tid;
  if (first && tid == 0 && found > a.prefill_seqs) atomicOr(a.err, kErrHint);
  fence_proxy_async();  // the scratch words are overwritten by TMA copies later
  __syncthreads();
  return *chosen_seq;
}

// A producer warp: streams the K (or V) tiles 0 .. ntiles-1 of sequence s, kv head g, keys
// [key_base, kend), into a ring of `stages` stages of kKVBytes each.  Each 16-token unit is found
// through the block table and fetched as 128-byte-swizzled TMA boxes (one per 64 columns).
// read_once: no other CTA reads these K/V (one CTA per sequence and kv head), so their lines
// enter L2 as the first to evict; the two-tile kernel's CTAs share every tile and keep the default.
// Before returning it waits (bounded) for its last copies, so none lands after the CTA retires.
template <int D, int BS, int kKeys>
__device__ __forceinline__ void produce_kv(const AttnArgs& a, const CUtensorMap* map, int s, int g,
                                           int kend, int ntiles, int stages, uint64_t* full,
                                           uint64_t* empty, uint32_t ring, int key_base,
                                           bool read_once) {
  constexpr int kUnits = kKeys / 16, kHalves = D / 64, kKVBytes = kHalves * kKeys * 128;
  const int lane = threadIdx.x & 31;
  // Block id of unit `lane` of tile j (0 past the keys).  The ids of tile j + 1 are loaded while
  // tile j waits for its stage, so the table read is off the copy's critical path.
  auto unit_block = [&](int j) {
    const int key0 = key_base + j * kKeys;
    const int units = min(kUnits, (kend - key0 + 15) >> 4);
    return lane < units
               ? a.block_tables[static_cast<int64_t>(s) * a.bt_stride + (key0 + 16 * lane) / BS]
               : 0;
  };
  const uint64_t pol = l2_policy_evict_first();  // for K/V no other CTA reads
  int issued = 0;
  int id_next = ntiles > 0 ? unit_block(0) : 0;
  for (int j = 0; j < ntiles; ++j) {
    const int st = j % stages, round = j / stages;
    const int id = id_next;
    if (j + 1 < ntiles) id_next = unit_block(j + 1);
    bool ok = true;
    if (lane == 0 && round > 0) ok = mbar_wait(smem_addr(&empty[st]), (round - 1) & 1,
                                               a.err, a.wait_limit_ns);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
    const int key0 = key_base + j * kKeys;
    const int units = min(kUnits, (kend - key0 + 15) >> 4);
    const uint32_t bar = smem_addr(&full[st]);
    if (lane == 0) mbar_arrive_expect_tx(bar, units * kHalves * 2048);
    const uint32_t dst = ring + st * kKVBytes;
    for (int u = 0; u < units; ++u) {
      const int blk = __shfl_sync(0xffffffffu, id, u);
      if (lane == 0) {
        const int y = (blk * a.num_kv_heads + g) * BS + ((key0 + 16 * u) % BS);
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          if (read_once)
            tma_load_2d_hint(dst + h * (kKeys * 128) + u * 2048, map, h * 64, y, bar, pol);
          else
            tma_load_2d(dst + h * (kKeys * 128) + u * 2048, map, h * 64, y, bar);
        }
      }
    }
    issued = j + 1;
  }
  if (lane == 0)
    for (int j = max(0, issued - stages); j < issued; ++j)
      mbar_wait(smem_addr(&full[j % stages]), (j / stages) & 1, a.err, a.wait_limit_ns);
}

// Widen, in place, key rows [32 p0, 32 p1) of a landed tile of E4M3 codes (stage at `dst`, the
// codes in its upper half) into the tile's fp16 layout, one key row per lane (see below).
template <int D, int kKeys>
__device__ __forceinline__ void widen_rows_f8(uint32_t dst, int rows, int p0, int p1) {
  constexpr int kKVBytes = (D / 64) * kKeys * 128, kCodes = kKVBytes / 2, kChunks = D / 16;
  const int lane = threadIdx.x & 31;
  for (int k0 = 32 * p0; k0 < rows && k0 < 32 * p1; k0 += 32) {
    const int k = k0 + lane;
    uint32_t w[kChunks][4];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const uint32_t src = dst + kCodes +
                           (D == 128 ? k * 128 + ((c ^ (k & 7)) << 4) : k * 64 + c * 16);
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[c][0]), "=r"(w[c][1]), "=r"(w[c][2]), "=r"(w[c][3])
                   : "r"(src)
                   : "memory");
    }
    if (D == 64) __syncwarp();  // rows 2k - 128, 2k - 127 may belong to other lanes
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int e8 = (c * 16 % 64) / 8;  // first 8-column chunk of dims c*16 .. c*16+15
      const uint32_t row = dst + (c * 16 / 64) * (kKeys * 128) + k * 128;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         row + (((e8 + q) ^ (k & 7)) << 4)),
                     "r"(f16x2_from_e4m3x2(w[c][2 * q])),
                     "r"(f16x2_from_e4m3x2(w[c][2 * q] >> 16)),
                     "r"(f16x2_from_e4m3x2(w[c][2 * q + 1])),
                     "r"(f16x2_from_e4m3x2(w[c][2 * q + 1] >> 16))
                     : "memory");
    }
    if (D == 64) __syncwarp();  // this pass's stores are done before the next pass loads
  }
}

// The same producer over an FP8 (E4M3) pool (read_once as above), with no extra shared memory:
// a tile's codes (16-row TMA boxes of D bytes, 128-byte swizzled for D = 128, plain 64-byte rows
// for D = 64) land in the upper half of the tile's own fp16 stage, completing on the stage's `land`
// barrier, and the warp widens them in place (exact: every E4M3 value is an fp16 value) into
// the 128-byte-swizzled [64-column chunk][key][128 B] layout of an fp16 tile, one key row per
// lane.  In place is safe: for D = 128 row k's fp16 bytes cover exactly row k's own codes,
// which its lane has loaded before it stores; for D = 64 they cover code rows 2k - 128 and
// 2k - 127, never above k, and every lane of a pass loads its row before any lane stores.
// Tile j + 1's copy is issued before tile j is widened, so the copy's latency overlaps the
// widening; then a proxy fence and all 32 lanes arrive on the stage's `full` barrier (count
// 32).  The scales are applied by the kernel (k_scale in the score scale, v_scale on the
// output).
// Passes (32 key rows each) of a 128-key tile the producer widens itself; for D = 128 a helper
// warp widens the rest of each K and V tile (rows never overlap another row's codes there).
template <int D>
constexpr int kF8MainPasses = D == 128 ? 2 : 4;

// The helper warp of an FP8 launch with D = 128: widens passes 2 and 3 of every K tile and every
// V tile in the order the MMA issuer consumes them (K_j, then V_j), each after the tile's codes
// landed, and arrives on the stage's `full` barrier (which then counts 64 arrivals).
template <int D, int kKeys>
__device__ __forceinline__ void widen_helper_f8(const AttnArgs& a, int kend, int ntiles,
                                                int key_base, int k_stages, int v_stages,
                                                uint32_t k_ring, uint32_t v_ring,
                                                uint64_t* k_full, uint64_t* v_full,
                                                uint64_t (*land)[3]) {
  constexpr int kKVBytes = (D / 64) * kKeys * 128;
  for (int j = 0; j < ntiles; ++j) {
    const int rows = min(kKeys / 16, (kend - (key_base + j * kKeys) + 15) >> 4) * 16;
    for (int t = 0; t < 2; ++t) {  // K, then V
      const int stages = t == 0 ? k_stages : v_stages, st = j % stages;
      const bool ok = mbar_wait(smem_addr(&land[t][st]), (j / stages) & 1, a.err, a.wait_limit_ns);
      if (!__all_sync(0xffffffffu, ok)) return;
      widen_rows_f8<D, kKeys>((t == 0 ? k_ring : v_ring) + st * kKVBytes, rows,
                              kF8MainPasses<D>, 4);
      fence_proxy_async();
      mbar_arrive(smem_addr(&(t == 0 ? k_full : v_full)[st]));
    }
  }
}

template <int D, int BS, int kKeys>
__device__ __forceinline__ void produce_kv_f8(const AttnArgs& a, const CUtensorMap* map, int s,
                                              int g, int kend, int ntiles, int stages,
                                              uint64_t* full, uint64_t* empty, uint32_t ring,
                                              uint64_t* land, int key_base, bool read_once) {
  constexpr int kUnits = kKeys / 16, kKVBytes = (D / 64) * kKeys * 128, kUnit8 = 16 * D;
  constexpr int kCodes = kKVBytes / 2;  // where a stage's codes land
  const int lane = threadIdx.x & 31;
  auto units_of = [&](int j) { return min(kUnits, (kend - (key_base + j * kKeys) + 15) >> 4); };
  auto unit_block = [&](int j) {
    const int key0 = key_base + j * kKeys;
    return lane < units_of(j)
               ? a.block_tables[static_cast<int64_t>(s) * a.bt_stride + (key0 + 16 * lane) / BS]
               : 0;
  };
  const uint64_t pol = l2_policy_evict_first();  // for K/V no other CTA reads
  // tile j's codes -> the upper half of its stage, completing on land[stage]
  auto fetch = [&](int j, int id) {
    const int st = j % stages, key0 = key_base + j * kKeys, units = units_of(j);
    const uint32_t bar = smem_addr(&land[st]);
    const uint32_t dst = ring + st * kKVBytes + kCodes;
    if (lane == 0) mbar_arrive_expect_tx(bar, units * kUnit8);
    for (int u = 0; u < units; ++u) {
      const int blk = __shfl_sync(0xffffffffu, id, u);
      if (lane == 0) {
        const int y = (blk * a.num_kv_heads + g) * BS + ((key0 + 16 * u) % BS);
        if (read_once)
          tma_load_2d_hint(dst + u * kUnit8, map, 0, y, bar, pol);
        else
          tma_load_2d(dst + u * kUnit8, map, 0, y, bar);
      }
    }
  };
  // tile j (landed) widened in place; false when a wait gave up
  auto widen = [&](int j) -> bool {
    const int st = j % stages;
    const bool ok = mbar_wait(smem_addr(&land[st]), (j / stages) & 1, a.err, a.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) return false;
    widen_rows_f8<D, kKeys>(ring + st * kKVBytes, units_of(j) * 16, 0, kF8MainPasses<D>);
    fence_proxy_async();  // the generic stores -> visible to the MMA's shared-memory reads
    mbar_arrive(smem_addr(&full[st]));
    return true;
  };
  int fetched = 0;
  int id_next = ntiles > 0 ? unit_block(0) : 0;
  bool ok = true;
  for (int j = 0; j < ntiles && ok; ++j) {
    const int st = j % stages, round = j / stages;
    const int id = id_next;
    if (j + 1 < ntiles) id_next = unit_block(j + 1);
    ok = round == 0 || mbar_wait(smem_addr(&empty[st]), (round - 1) & 1, a.err, a.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    fetch(j, id);
    fetched = j + 1;
    if (j >= 1) ok = widen(j - 1);
  }
  if (ok && ntiles > 0) widen(ntiles - 1);
  // copies requested but never widened (a wait gave up) must land before the CTA retires
  if (lane == 0)
    for (int j = max(0, fetched - stages); j < fetched; ++j)
      mbar_wait(smem_addr(&land[j % stages]), (j / stages) & 1, a.err, a.wait_limit_ns);
}

// F8: the pool holds E4M3 codes, widened in place in the fp16 stages (no extra memory).
template <int D, bool F8 = false>
struct PairCfg {
  static constexpr int kRows = 128;  // MMA M: (query token, head) rows of one Q tile
  static constexpr int kQTiles = 2;  // Q tiles per CTA, sharing every K/V tile
  static constexpr int kKeys = 128;  // keys per K/V tile: N of S, K of P V
  static constexpr int kHalves = D / 64;                  // 128-byte column chunks of a row
  static constexpr int kHalfBytes = kRows * 128;          // one 64-column chunk of a 128-row tile
  static constexpr int kQBytes = kHalves * kHalfBytes;    // one Q tile, [half][row][128 B]
  static constexpr int kKVBytes = kHalves * kKeys * 128;  // K (or V) tile, [half][key][128 B]
  static constexpr int kKStages = 2;
  static constexpr int kVStages = 3;
  static constexpr int kSmemBytes =
      kQTiles * kQBytes + (kKStages + kVStages) * kKVBytes + 1024;
  // Two warpgroups per Q tile: one per half of each key tile's columns (and of O's columns),
  // so a row's softmax is shared by two threads that trade their maxima once per key tile.
  static constexpr int kSoftmax = 512;
  static constexpr int kPerTile = 256;                    // softmax threads of one Q tile
  // + a warpgroup of K producer, V producer, MMA issuer and one idle warp
  static constexpr int kThreads = kSoftmax + 4 * 32;
  // Registers: launched at 96 per thread (640 x 96 = 61440); the producer warpgroup gives back
  // down to 64 and the four softmax warpgroups take 104: 512 x 104 + 128 x 64 = 61440.
  static constexpr int kLaunchRegs = 96;
  static constexpr int kRegsSoftmax = 104;
  static constexpr int kRegsOther = 64;
  // TMEM columns: S/P of Q tile A [0,128), of Q tile B [128,256), O_A, O_B from 256.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
  static_assert(kQTiles * kKeys + kQTiles * D <= 512, "S/P buffers and accumulators fit TMEM");
  static_assert(kSmemBytes + 1024 <= 232448, "dynamic + static shared memory fit one SM");
  static constexpr float kRescaleLog2 = 8.f;              // raise the max only past 2^8
};

// CASCADE: the shared-prefix pass.  Rows are every query row of the batch (all decode rows,
// row i of q), keys are the cascade_span 512-key partitions blockIdx.z * cascade_span .. of the
// prefix that every sequence shares (read through sequence 0's table), no causal mask; the
// epilogue writes the rows' partials (m, l, O / l) for the log-sum-exp merge into the slot of
// the first of those partitions instead of the output.
template <int D, int BS, bool CASCADE, bool BF, bool F8>
__global__ void __launch_bounds__(PairCfg<D>::kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = PairCfg<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  __shared__ __align__(8) uint64_t v_full[C::kVStages], v_empty[C::kVStages];
  // Per Q tile: S_t(j + 1) is issued only after P_t V_j, which waits for the softmax's P_t(j),
  // so each of these runs at most one phase ahead of its waiter (no parity ambiguity).
  __shared__ __align__(8) uint64_t s_full[C::kQTiles], p_full[C::kQTiles];
  __shared__ __align__(8) uint64_t q_full, drain;
  __shared__ __align__(8) uint64_t land[2][3];  // F8: [K / V][stage] codes landed
  __shared__ uint32_t tmem_base;
  __shared__ int warp_count[C::kThreads / 32];
  __shared__ int chosen_seq;
  // [Q tile][column half][row]: each half's key-tile maximum, rounded up to bfloat16 (so both
  // halves of a row take the same base from the same two stored values)
  __shared__ __nv_bfloat16 half_max[C::kQTiles][2][C::kRows];

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t q_s = smem_addr(smem);                     // Q tiles A, B
  const uint32_t k_s = q_s + C::kQTiles * C::kQBytes;       // K ring
  const uint32_t v_s = k_s + C::kKStages * C::kKVBytes;     // V ring
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Work item (q-tile pair x, kv head g, prefill sequence z): the grid's coordinates, or, when
  // the launch is one of a series that each cover a slice of the items, item_base + blockIdx.x
  // decoded in the same (x fastest, then g, then z) order.
  int bx = blockIdx.x, g = blockIdx.y, bz = blockIdx.z, nx = gridDim.x;
  if (!CASCADE && a.items_x > 0) {
    const int item = a.item_base + static_cast<int>(blockIdx.x);
    nx = a.items_x;
    bx = item % nx;
    g = (item / nx) % a.num_kv_heads;
    bz = item / (nx * a.num_kv_heads);
  }
  const int tile_q = C::kRows / a.group;  // query tokens per Q tile
  int s, qt, row0, q_len, ctx, key_base = 0;
  int tiles[C::kQTiles];
  int kend, ntiles;  // keys loaded: [key_base, kend), in ntiles 128-key tiles
  if constexpr (CASCADE) {
    s = 0;
    qt = blockIdx.x;
    row0 = 0;
    q_len = static_cast<int>(a.num_tokens);
    key_base = blockIdx.z * a.cascade_span * kPartitionTokens;
    ctx = 0;  // unused: no causal mask inside the shared prefix
    kend = key_base + a.cascade_span * kPartitionTokens;
    ntiles = a.cascade_span * kPartitionTokens / C::kKeys;
    if (qt * C::kQTiles * tile_q >= q_len) return;
#pragma unroll
    for (int t = 0; t < C::kQTiles; ++t)
      tiles[t] = qt * C::kQTiles * tile_q + t * tile_q < q_len ? ntiles : 0;
  } else {
    // Later q tiles of a chunk see more keys: dispatch them first so the grid's tail is short.
    qt = nx - 1 - bx;
    s = find_prefill_seq<C::kThreads>(a, warp_count, &chosen_seq, bz, bx == 0 && g == 0 && bz == 0);
    if (s < 0) return;
    row0 = a.query_start_loc[s];
    q_len = a.query_start_loc[s + 1] - row0;
    if (q_len <= 1) return;  // decode rows and idle sequences are handled elsewhere
    const int L = a.seq_lens[s];
    if (q_len > L || (L + BS - 1) / BS > a.max_blocks || row0 < 0 ||
        row0 + q_len > a.num_tokens) {
      if (qt == 0 && tid == 0) atomicOr(a.err, kErrDescriptor);
      return;
    }
    if ((q_len + C::kQTiles * tile_q - 1) / (C::kQTiles * tile_q) > nx) {
      if (qt == 0 && tid == 0) atomicOr(a.err, kErrHint);
      return;
    }
    if (qt * C::kQTiles * tile_q >= q_len) return;
    ctx = L - q_len;
    // Key tiles of each Q tile: keys [0, ctx + last row + 1); Q tile B may hold no row at all.
#pragma unroll
    for (int t = 0; t < C::kQTiles; ++t) {
      const int first = qt * C::kQTiles * tile_q + t * tile_q;
      tiles[t] = first < q_len
                     ? (ctx + min(q_len, first + tile_q) + C::kKeys - 1) / C::kKeys
                     : 0;
    }
    kend = ctx + min(q_len, qt * C::kQTiles * tile_q + C::kQTiles * tile_q);
    ntiles = (kend + C::kKeys - 1) / C::kKeys;  // == max over Q tiles
  }
  const int qbase = qt * C::kQTiles * tile_q;

  // Every block id the CTA will read is checked before any copy is issued.
  int bad = 0;
  const int nblk = (kend + BS - 1) / BS;
  for (int j = key_base / BS + tid; j < nblk; j += C::kThreads) {
    const int32_t blk = a.block_tables[static_cast<int64_t>(s) * a.bt_stride + j];
    if (blk < 0 || blk >= a.num_blocks) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(a.err, kErrBlockRange);
    return;
  }

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int st = 0; st < C::kKStages; ++st) {
      mbar_init(smem_addr(&k_full[st]), F8 ? (D == 128 ? 64 : 32) : 1);
      mbar_init(smem_addr(&k_empty[st]), 1);
    }
    for (int st = 0; st < C::kVStages; ++st) {
      mbar_init(smem_addr(&v_full[st]), F8 ? (D == 128 ? 64 : 32) : 1);
      mbar_init(smem_addr(&v_empty[st]), 1);
    }
    for (int t = 0; t < C::kQTiles; ++t) {
      mbar_init(smem_addr(&s_full[t]), 1);
      mbar_init(smem_addr(&p_full[t]), C::kPerTile);
    }
    mbar_init(smem_addr(&q_full), C::kSoftmax);
    mbar_init(smem_addr(&drain), 1);
    for (int b = 0; b < 6; ++b) mbar_init(smem_addr(&land[b / 3][b % 3]), 1);
    mbar_init_fence();
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = tmem_base;

  constexpr int kKWarp = C::kSoftmax / 32, kVWarp = kKWarp + 1, kMmaWarp = kKWarp + 2;
  static_assert(C::kRegsSoftmax * C::kSoftmax + C::kRegsOther * (C::kThreads - C::kSoftmax) <=
                    C::kLaunchRegs * C::kThreads,
                "register split exceeds the launch allocation");
  if (warp >= kKWarp) {
  // ================================================ producer / MMA warpgroup (warps 16-19)
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsOther));
  if (warp == kKWarp || warp == kVWarp) {
    // ============================================================== producer warps (K, V)
    const bool is_v = warp == kVWarp;
    if constexpr (F8)
      produce_kv_f8<D, BS, C::kKeys>(a, is_v ? &vmap : &kmap, s, g, kend, ntiles,
                                     is_v ? C::kVStages : C::kKStages, is_v ? v_full : k_full,
                                     is_v ? v_empty : k_empty, is_v ? v_s : k_s,
                                     land[is_v ? 1 : 0], key_base, false);
    else
      produce_kv<D, BS, C::kKeys>(a, is_v ? &vmap : &kmap, s, g, kend, ntiles,
                                  is_v ? C::kVStages : C::kKStages, is_v ? v_full : k_full,
                                  is_v ? v_empty : k_empty, is_v ? v_s : k_s, key_base, false);
  } else if (warp == kMmaWarp && lane == 0) {
    // ============================================================== MMA issuer (one thread)
    constexpr uint32_t kIdS = umma_idesc_f16(C::kRows, C::kKeys, 0, 0, BF);
    constexpr uint32_t kIdO = umma_idesc_f16(C::kRows, D, 0, 1, BF);
    // S_t(j) = Q_t K_j^T into TMEM buffer t (K stage j must have landed).
    auto issue_s = [&](int t, int j) {
      const uint32_t kst = k_s + (j % C::kKStages) * C::kKVBytes;
      const uint32_t qb = q_s + t * C::kQBytes;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * C::kHalfBytes + (k & 3) * 32;
        umma_f16(tmem + t * C::kKeys, umma_sdesc(qb + off, 16, 1024),
                 umma_sdesc(kst + (k >> 2) * (C::kKeys * 128) + (k & 3) * 32, 16, 1024), kIdS,
                 k > 0);
      }
      umma_commit(smem_addr(&s_full[t]));
    };
    // O_t += P_t V_j (V stage j must have landed, P_t(j) must be written).
    auto issue_pv = [&](int t, int j) {
      const uint32_t vb = v_s + (j % C::kVStages) * C::kKVBytes;
#pragma unroll
      for (int k = 0; k < C::kKeys / 16; ++k)
        umma_f16_tmem_a(tmem + C::kOCol + t * D, tmem + t * C::kKeys + k * 8,
                        umma_sdesc(vb + k * 16 * 128, C::kKeys * 128, 1024), kIdO,
                        (j > 0 || k > 0));
    };
    auto kwait = [&](int j) {
      const bool ok = mbar_wait(smem_addr(&k_full[j % C::kKStages]), (j / C::kKStages) & 1,
                                a.err, a.wait_limit_ns);
      tmem_fence_after_sync();
      return ok;
    };
    bool ok = mbar_wait(smem_addr(&q_full), 0, a.err, a.wait_limit_ns) && kwait(0);
    if (ok) {
#pragma unroll
      for (int t = 0; t < C::kQTiles; ++t)
        if (tiles[t] > 0) issue_s(t, 0);
      umma_commit(smem_addr(&k_empty[0]));
    }
    for (int j = 0; ok && j < ntiles; ++j) {
      const int vst = j % C::kVStages;
      const bool more = j + 1 < ntiles;
      ok = mbar_wait(smem_addr(&v_full[vst]), (j / C::kVStages) & 1, a.err, a.wait_limit_ns);
      bool k_ready = false;  // K_{j+1} is waited for just before its first use
#pragma unroll
      for (int t = 0; ok && t < C::kQTiles; ++t) {
        if (j >= tiles[t]) continue;
        ok = mbar_wait(smem_addr(&p_full[t]), j & 1, a.err, a.wait_limit_ns);
        if (!ok) break;
        tmem_fence_after_sync();
        issue_pv(t, j);
        // V_j's stage is free once the last P V that reads it is done: release it before the
        // next S so the producer can start the refill sooner.
        if (t == C::kQTiles - 1 || j >= tiles[t + 1]) umma_commit(smem_addr(&v_empty[vst]));
        if (j + 1 < tiles[t]) {
          if (!k_ready) {
            ok = kwait(j + 1);
            k_ready = true;
            if (!ok) break;
          }
          issue_s(t, j + 1);
        }
      }
      if (!ok) break;
      if (more) umma_commit(smem_addr(&k_empty[(j + 1) % C::kKStages]));
    }
    // Every MMA this thread issued has finished before O is read or the CTA tears down.
    umma_commit(smem_addr(&drain));
    mbar_wait(smem_addr(&drain), 0, a.err, a.wait_limit_ns);
  } else if (F8 && D == 128 && warp == kMmaWarp + 1) {
    // ============================================================== FP8 widening helper
    widen_helper_f8<D, C::kKeys>(a, kend, ntiles, key_base, C::kKStages, C::kVStages, k_s, v_s,
                                 k_full, v_full, land);
  }  // lanes 1-31 of warp 18 have no role (warp 19 neither, unless it helps widen FP8 tiles)
  } else {
    // ============================================================== softmax warps 0-15
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsSoftmax));
    // Warp w: Q tile t = w / 8, column half h = (w / 4) % 2 (keys 64h .. 64h + 63 of every key
    // tile and O columns h D / 2 .. of the output), TMEM lanes 32 (w % 4) .. + 31, one row per
    // thread.  The two warps of a row quarter meet at named barrier 1 + 4 t + w % 4 once per key
    // tile (trading their maxima) and once in the epilogue (trading their sums); every meeting
    // also ORs the pair's failed waits, so both leave together and neither waits alone.
    constexpr int kHalfKeys = C::kKeys / 2, kHalfD = D / 2;
    const int t = warp >> 3;                  // Q tile of this warp
    const int h = (warp >> 2) & 1;            // column half
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;        // TMEM lane = row of the Q tile
    const uint32_t pair_bar = 1 + t * 4 + quarter;
    const int qi = r / a.group, hg = r % a.group;
    const int first = qbase + t * tile_q;     // first query token of the Q tile
    const int tok = first + qi;
    const bool rv = qi < tile_q && tok < q_len;
    const int pos = ctx + (rv ? tok : first);  // padding rows mirror the tile's first row
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t sbuf = tmem + lane_addr + t * C::kKeys;
    const uint32_t obuf = tmem + lane_addr + C::kOCol + t * D + h * kHalfD;
    const int my_tiles = tiles[t];
    // The V rows past kend are zeroed by the Q tile whose P V of the last key tile comes first.
    const bool zeroes_v = !CASCADE && (t == 0 ? tiles[0] == ntiles : tiles[0] < ntiles);

    // Half h of the Q row -> shared memory, 128B-swizzled K-major.
    {
      const __half* qrow = a.q + static_cast<int64_t>(row0 + (rv ? tok : 0)) * a.q_stride +
                           static_cast<int64_t>(g * a.group + hg) * D;
      const uint32_t qb = q_s + t * C::kQBytes;
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {
        const int c = h * (D / 16) + cc;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rv) v = __ldg(reinterpret_cast<const uint4*>(qrow + c * 8));
        const uint32_t dst = qb + (c >> 3) * C::kHalfBytes + swz128(r, c & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async();
      mbar_arrive(smem_addr(&q_full));
    }

    bool stopped = false;  // a wait of this pair of threads gave up
    float m_run = -INFINITY, l_run = 0.f;
    const int min_pos = ctx + first;
    const bool prescale = !(a.scale_log2 > 0.f);
    const float mul = prescale ? 1.f : a.scale_log2;  // exponent = fma(score, mul, -m)
    for (int j = 0; j < my_tiles; ++j) {
      // S_t(j) done; it was issued after P_t V_{j-1}, so O_t is settled too.
      const bool got = mbar_wait(smem_addr(&s_full[t]), j & 1, a.err, a.wait_limit_ns);
      uint32_t sv[kHalfKeys / 32][32];
      float mloc = -INFINITY;
      const int key0 = j * C::kKeys + h * kHalfKeys;
      if (got) {
        tmem_fence_after_sync();
#pragma unroll
        for (int qq = 0; qq < kHalfKeys / 32; ++qq)
          tmem_ld32(sbuf + h * kHalfKeys + qq * 32, sv[qq]);
        tmem_wait_ld();
#pragma unroll
        for (int qq = 0; qq < kHalfKeys / 32; ++qq) tmem_regs_ready(sv[qq]);
        // Scores stay raw where scale > 0 (the max commutes with the scale, which is folded
        // into the exponent's FMA below); otherwise they are scaled here.  Masked keys: -inf.
        const bool masked = !CASCADE && key0 + kHalfKeys - 1 > min_pos;
        if (prescale || masked) {
#pragma unroll
          for (int c = 0; c < kHalfKeys; ++c) {
            float v = __uint_as_float(sv[c >> 5][c & 31]);
            if (prescale) v *= a.scale_log2;
            if (masked && key0 + c > pos) v = -INFINITY;
            sv[c >> 5][c & 31] = __float_as_uint(v);
          }
        }
        float m2[2] = {-INFINITY, -INFINITY};  // two chains of three-input maxima
#pragma unroll
        for (int c = 0; c < kHalfKeys; c += 2)
          m2[(c >> 1) & 1] = fmax3(m2[(c >> 1) & 1], __uint_as_float(sv[c >> 5][c & 31]),
                                   __uint_as_float(sv[c >> 5][(c & 31) + 1]));
        mloc = fmaxf(m2[0], m2[1]);
      }
      // Trade maxima: rounded up, the stored value is >= the half's max, and both threads read
      // the same two values, so they take the same base.  This half's S columns have been read
      // (wait::ld above) before the other half may store P over them (after the barrier).
      half_max[t][h][r] = __float2bfloat16_ru(mloc);
      tmem_fence_before_sync();
      if (bar_sync_or(pair_bar, 64, !got)) {
        stopped = true;
        break;
      }
      tmem_fence_after_sync();
      const float mx = fmaxf(__bfloat162float(half_max[t][0][r]),
                             __bfloat162float(half_max[t][1][r])) * mul;
      float alpha = 1.f;
      if (mx > m_run + C::kRescaleLog2 || (m_run == -INFINITY && mx > -INFINITY)) {
        alpha = ex2_approx(m_run - mx);  // 0 when m_run is still -inf
        m_run = mx;
      }
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c0 = 0; c0 < kHalfD; c0 += 8) {
          uint32_t tt[8];
          tmem_ld8(obuf + c0, tt);
          tmem_wait_ld();
          tmem_regs_ready(tt);
#pragma unroll
          for (int c = 0; c < 8; ++c) tt[c] = __float_as_uint(__uint_as_float(tt[c]) * alpha);
          tmem_st8(obuf + c0, tt);
        }
      }

      // P (fp16) of this half's keys -> TMEM columns h * 32 .. + 31 of the buffer, two keys per
      // column; l keeps the unrounded p.  A row with every key so far masked keeps m = -inf and
      // gets p = 0.
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      // exponents and sums two keys at a time (packed fp32 pairs: the same roundings as fmaf
      // and + per key)
      const uint64_t mul2 = f32x2(mul, mul), negm2 = f32x2(neg_m, neg_m);
      uint64_t ps2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
      for (int q8 = 0; q8 < kHalfKeys / 16; ++q8) {  // 16 keys -> 8 columns of P at a time
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int k = q8 * 16 + 2 * c;
          float x0, x1;
          f32x2_split(ffma2(f32x2(__uint_as_float(sv[k >> 5][k & 31]),
                                  __uint_as_float(sv[k >> 5][(k & 31) + 1])),
                            mul2, negm2),
                      x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          ps2[c & 1] = fadd2(ps2[c & 1], f32x2(p0, p1));
          pk[c] = pack2<BF>(p0, p1);
        }
        tmem_st8(sbuf + h * (kHalfKeys / 2) + q8 * 8, pk);
      }
      float s0, s1, s2, s3;
      f32x2_split(ps2[0], s0, s1);
      f32x2_split(ps2[1], s2, s3);
      l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));

      const int tile0 = j * C::kKeys;
      if (zeroes_v && j == ntiles - 1 && tile0 + C::kKeys > kend) {
        // The last key tile: V rows at or past kend may be stale or NaN; zero them once the
        // tile has landed (the MMA reads V only after p_full below).  The thread of row r and
        // half h clears half h of V row r (its 64-column chunk; D = 64 has one chunk).
        const int vst = j % C::kVStages;
        const bool landed =
            mbar_wait(smem_addr(&v_full[vst]), (j / C::kVStages) & 1, a.err, a.wait_limit_ns);
        if (landed && tile0 + r >= kend && h < C::kHalves) {
          const uint32_t vrow = v_s + vst * C::kKVBytes + h * (C::kKeys * 128) + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(vrow + c * 16),
                         "r"(0u), "r"(0u), "r"(0u), "r"(0u)
                         : "memory");
        }
        fence_proxy_async();
        if (!landed) stopped = true;  // the last tile: the epilogue's meeting ends both
      }
      if (stopped) break;
      tmem_wait_st();
      tmem_fence_before_sync();
      mbar_arrive(smem_addr(&p_full[t]));
    }

    // Epilogue: O_t / l -> out (fp16, rows of real query tokens only); the shared-prefix pass
    // writes the rows' partials of its prefix partitions instead: m (log2 units), l and O / l.
    // The two halves' sums are traded through the Q tile's shared memory, which no MMA reads
    // once `drain` has completed.
    bool ok = !stopped && my_tiles > 0;
    if (ok) ok = mbar_wait(smem_addr(&drain), 0, a.err, a.wait_limit_ns);
    float* l_half = reinterpret_cast<float*>(smem) + (t * 2 + h) * C::kRows;
    if (ok) l_half[r] = l_run;
    if (!bar_sync_or(pair_bar, 64, !ok)) {
      const float l_all = l_run + reinterpret_cast<const float*>(smem)[(t * 2 + (h ^ 1)) *
                                                                      C::kRows + r];
      tmem_fence_after_sync();
      const float inv = a.v_scale / l_all;  // v_scale: 1, or the FP8 pool's V scale
      if constexpr (CASCADE) {
        const int64_t pidx =
            (static_cast<int64_t>(row0 + tok) * a.num_q_heads + g * a.group + hg) * a.max_parts +
            blockIdx.z * a.cascade_span;
        if (rv && h == 0) {
          a.part_m[pidx] = m_run;
          a.part_l[pidx] = l_all;
        }
#pragma unroll
        for (int c0 = 0; c0 < kHalfD; c0 += 16) {
          uint32_t tt[16];
          tmem_ld16(obuf + c0, tt);
          tmem_wait_ld();
          tmem_regs_ready(tt);
          if (rv) {
#pragma unroll
            for (int c = 0; c < 16; c += 4)
              *reinterpret_cast<float4*>(a.part_o + pidx * D + h * kHalfD + c0 + c) =
                  make_float4(__uint_as_float(tt[c]) * inv, __uint_as_float(tt[c + 1]) * inv,
                              __uint_as_float(tt[c + 2]) * inv, __uint_as_float(tt[c + 3]) * inv);
          }
        }
      } else {
        __half* dst = a.out + (static_cast<int64_t>(row0 + tok) * a.num_q_heads + g * a.group +
                               hg) * D + h * kHalfD;
#pragma unroll
        for (int c0 = 0; c0 < kHalfD; c0 += 16) {
          uint32_t tt[16];
          tmem_ld16(obuf + c0, tt);
          tmem_wait_ld();
          tmem_regs_ready(tt);
          if (rv) {
#pragma unroll
            for (int c = 0; c < 16; c += 8) {
              uint4 v;
              v.x = pack2<BF>(__uint_as_float(tt[c]) * inv, __uint_as_float(tt[c + 1]) * inv);
              v.y = pack2<BF>(__uint_as_float(tt[c + 2]) * inv, __uint_as_float(tt[c + 3]) * inv);
              v.z = pack2<BF>(__uint_as_float(tt[c + 4]) * inv, __uint_as_float(tt[c + 5]) * inv);
              v.w = pack2<BF>(__uint_as_float(tt[c + 6]) * inv, __uint_as_float(tt[c + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + c0 + c) = v;
            }
          }
        }
      }
    }
  }

  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
}

template <int D, bool F8 = false>
struct ParityCfg {
  static constexpr int kRows = 128;  // MMA M: (query token, head) rows of the tile
  static constexpr int kKeys = 128;  // keys per K/V tile: N of S, K of P V
  static constexpr int kHalves = D / 64;                  // 128-byte column chunks of a row
  static constexpr int kHalfBytes = kRows * 128;          // one 64-column chunk of a 128-row tile
  static constexpr int kQBytes = kHalves * kHalfBytes;    // [half][row][128 B]
  static constexpr int kKVBytes = kHalves * kKeys * 128;  // K (or V) tile, [half][key][128 B]
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kSmemBytes = kQBytes + (kKStages + kVStages) * kKVBytes + 1024;
  // the kernel's static shared memory (barriers, the two parities' m and l per row) is ~2.3 KB
  static_assert(kSmemBytes + 2560 <= 232448, "dynamic + static shared memory fit one SM");
  static constexpr int kSoftmax = 256;                    // 8 softmax warps: 2 per row quarter
  static constexpr int kParity = 128;                     // softmax threads per key-tile parity
  // + a warpgroup of K producer, V producer, MMA issuer and one idle warp
  static constexpr int kThreads = kSoftmax + 4 * 32;
  // Registers: launched at 168 per thread (384 x 168 = 64512); the producer warpgroup gives
  // back down to 72 and the two softmax warpgroups take 216: 256 x 216 + 128 x 72 = 64512.
  static constexpr int kLaunchRegs = 168;
  static constexpr int kRegsSoftmax = 216;
  static constexpr int kRegsOther = 72;
  // TMEM columns: S/P of even tiles [0,128), of odd tiles [128,256), O_even, O_odd from 256.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
  static constexpr float kRescaleLog2 = 8.f;              // raise the max only past 2^8
};

// CASCADE: the shared-prefix pass, as in the pair kernel (rows: every query row of the batch;
// keys: prefix partitions blockIdx.z * cascade_span .. through sequence 0's table; partials out).
template <int D, int BS, bool CASCADE, bool BF, bool F8>
__global__ void __launch_bounds__(ParityCfg<D>::kThreads, 1)
    prefill_parity_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using C = ParityCfg<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  __shared__ __align__(8) uint64_t v_full[C::kVStages], v_empty[C::kVStages];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2];  // per key-tile parity
  __shared__ __align__(8) uint64_t q_full, drain;
  __shared__ __align__(8) uint64_t land[2][3];  // F8: [K / V][stage] codes landed
  __shared__ uint32_t tmem_base;
  __shared__ float red_m[2][128];  // [parity][row]: running max and sum for the final merge
  __shared__ float red_l[2][128];
  __shared__ int softmax_stop;  // set by a softmax thread whose wait gave up
  __shared__ int warp_count[ParityCfg<D>::kThreads / 32];
  __shared__ int chosen_seq;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t q_s = smem_addr(smem);
  const uint32_t k_s = q_s + C::kQBytes;                  // K ring
  const uint32_t v_s = k_s + C::kKStages * C::kKVBytes;   // V ring
  const int g = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_q = C::kRows / a.group;  // query tokens per CTA
  int s, qt, row0, q_len, ctx, kend, ntiles, key_base = 0;  // keys [key_base, kend)
  if constexpr (CASCADE) {
    s = 0;
    qt = blockIdx.x;
    row0 = 0;
    q_len = static_cast<int>(a.num_tokens);
    ctx = 0;  // unused: no causal mask inside the shared prefix
    key_base = blockIdx.z * a.cascade_span * kPartitionTokens;
    kend = key_base + a.cascade_span * kPartitionTokens;
    ntiles = a.cascade_span * kPartitionTokens / C::kKeys;
    if (qt * tile_q >= q_len) return;
  } else {
    // Later q tiles of a chunk see more keys, and longer sequences more tiles: dispatch them
    // first so the grid's tail is short.
    qt = gridDim.x - 1 - blockIdx.x;
    s = find_prefill_seq_longest_first<C::kThreads>(
        a, warp_count, &chosen_seq, reinterpret_cast<int*>(smem), blockIdx.z,
        blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0);
    if (s < 0) return;
    row0 = a.query_start_loc[s];
    q_len = a.query_start_loc[s + 1] - row0;
    if (q_len <= 1) return;  // decode rows and idle sequences are handled elsewhere
    const int L = a.seq_lens[s];
    if (q_len > L || (L + BS - 1) / BS > a.max_blocks || row0 < 0 ||
        row0 + q_len > a.num_tokens) {
      if (qt == 0 && tid == 0) atomicOr(a.err, kErrDescriptor);
      return;
    }
    if ((q_len + tile_q - 1) / tile_q > static_cast<int>(gridDim.x)) {
      if (qt == 0 && tid == 0) atomicOr(a.err, kErrHint);
      return;
    }
    if (qt * tile_q >= q_len) return;
    ctx = L - q_len;
    kend = ctx + min(q_len, qt * tile_q + tile_q);  // keys [0, kend) are visible to some row
    ntiles = (kend + C::kKeys - 1) / C::kKeys;
  }
  const int qbase = qt * tile_q;

  // Every block id the CTA will read is checked before any copy is issued.
  int bad = 0;
  const int nblk = (kend + BS - 1) / BS;
  for (int j = key_base / BS + tid; j < nblk; j += C::kThreads) {
    const int32_t blk = a.block_tables[static_cast<int64_t>(s) * a.bt_stride + j];
    if (blk < 0 || blk >= a.num_blocks) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(a.err, kErrBlockRange);
    return;
  }

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int st = 0; st < C::kKStages; ++st) {
      mbar_init(smem_addr(&k_full[st]), F8 ? (D == 128 ? 64 : 32) : 1);
      mbar_init(smem_addr(&k_empty[st]), 1);
    }
    for (int st = 0; st < C::kVStages; ++st) {
      mbar_init(smem_addr(&v_full[st]), F8 ? (D == 128 ? 64 : 32) : 1);
      mbar_init(smem_addr(&v_empty[st]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&s_full[b]), 1);
      mbar_init(smem_addr(&p_full[b]), C::kParity);
    }
    mbar_init(smem_addr(&q_full), C::kSoftmax);
    mbar_init(smem_addr(&drain), 1);
    for (int b = 0; b < 6; ++b) mbar_init(smem_addr(&land[b / 3][b % 3]), 1);
    mbar_init_fence();
    softmax_stop = 0;
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = tmem_base;

  constexpr int kKWarp = C::kSoftmax / 32, kVWarp = kKWarp + 1, kMmaWarp = kKWarp + 2;
  static_assert(C::kRegsSoftmax * C::kSoftmax + C::kRegsOther * (C::kThreads - C::kSoftmax) <=
                    C::kLaunchRegs * C::kThreads,
                "register split exceeds the launch allocation");
  if (warp >= kKWarp) {
  // ================================================ producer / MMA warpgroup (warps 8-11)
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsOther));
  if (warp == kKWarp || warp == kVWarp) {
    // ============================================================== producer warps (K, V)
    const bool is_v = warp == kVWarp;
    if constexpr (F8)
      produce_kv_f8<D, BS, C::kKeys>(a, is_v ? &vmap : &kmap, s, g, kend, ntiles,
                                     is_v ? C::kVStages : C::kKStages, is_v ? v_full : k_full,
                                     is_v ? v_empty : k_empty, is_v ? v_s : k_s,
                                     land[is_v ? 1 : 0], key_base,
                                     !CASCADE);
    else
      produce_kv<D, BS, C::kKeys>(a, is_v ? &vmap : &kmap, s, g, kend, ntiles,
                                  is_v ? C::kVStages : C::kKStages, is_v ? v_full : k_full,
                                  is_v ? v_empty : k_empty, is_v ? v_s : k_s, key_base,
                                  !CASCADE);
  } else if (warp == kMmaWarp && lane == 0) {
    // ============================================================== MMA issuer (one thread)
    // Issuing a tcgen05.mma waits until the pipe takes it and the pipe queues almost nothing,
    // so every other instruction of this thread idles the tensor cores for its duration: the
    // issuer runs alone, with no warp-collective operations.
    constexpr uint32_t kIdS = umma_idesc_f16(C::kRows, C::kKeys, 0, 0, BF);
    constexpr uint32_t kIdO = umma_idesc_f16(C::kRows, D, 0, 1, BF);
    // S_j = Q K_j^T into TMEM buffer j % 2; frees its K stage once done.
    auto issue_s = [&](int j) {
      const int st = j % C::kKStages;
      if (!mbar_wait(smem_addr(&k_full[st]), (j / C::kKStages) & 1,
                     a.err, a.wait_limit_ns)) return false;
      tmem_fence_after_sync();
      const uint32_t kst = k_s + st * C::kKVBytes;
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * C::kHalfBytes + (k & 3) * 32;
        umma_f16(tmem + (j & 1) * 128, umma_sdesc(q_s + off, 16, 1024),
                 umma_sdesc(kst + (k >> 2) * (C::kKeys * 128) + (k & 3) * 32, 16, 1024), kIdS,
                 k > 0);
      }
      umma_commit(smem_addr(&s_full[j & 1]));
      umma_commit(smem_addr(&k_empty[st]));
      return true;
    };
    bool ok = mbar_wait(smem_addr(&q_full), 0,
                        a.err, a.wait_limit_ns) && issue_s(0) && (ntiles < 2 || issue_s(1));
    for (int j = 0; ok && j < ntiles; ++j) {
      const int vst = j % C::kVStages;
      ok = mbar_wait(smem_addr(&p_full[j & 1]), (j >> 1) & 1, a.err, a.wait_limit_ns) &&
           mbar_wait(smem_addr(&v_full[vst]), (j / C::kVStages) & 1, a.err, a.wait_limit_ns);
      if (!ok) break;
      tmem_fence_after_sync();
      const uint32_t vb = v_s + vst * C::kKVBytes;
#pragma unroll
      for (int k = 0; k < C::kKeys / 16; ++k)
        umma_f16_tmem_a(tmem + C::kOCol + (j & 1) * D, tmem + (j & 1) * 128 + k * 8,
                        umma_sdesc(vb + k * 16 * 128, C::kKeys * 128, 1024), kIdO,
                        (j > 1 || k > 0));
      umma_commit(smem_addr(&v_empty[vst]));
      if (j + 2 < ntiles) ok = issue_s(j + 2);
    }
    // Every MMA this thread issued has finished before O is read or the CTA tears down.
    umma_commit(smem_addr(&drain));
    mbar_wait(smem_addr(&drain), 0, a.err, a.wait_limit_ns);
  } else if (F8 && D == 128 && warp == kMmaWarp + 1) {
    // ============================================================== FP8 widening helper
    widen_helper_f8<D, C::kKeys>(a, kend, ntiles, key_base, C::kKStages, C::kVStages, k_s, v_s,
                                 k_full, v_full, land);
  }  // warp 11 has no role unless it helps widen FP8 tiles
  } else {
    // ============================================================== softmax warps 0-7
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsSoftmax));
    // Warp w takes key tiles j with j % 2 == par = w / 4 for TMEM lanes 32(w%4) .. +31, one
    // row per thread, all columns.  Its O accumulator is O_par.
    constexpr int kOHalf = D / 2;             // output columns per thread in the epilogue
    const int par = warp >> 2;
    const int r = (warp & 3) * 32 + lane;     // TMEM lane = tile row
    const int qi = r / a.group, hg = r % a.group;
    const bool rv = qi < tile_q && qbase + qi < q_len;
    const int pos = ctx + (rv ? qbase + qi : qbase);  // padding rows mirror the first row
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t obuf = tmem + lane_addr + C::kOCol + par * D;

    // Half par of the Q row -> shared memory, 128B-swizzled K-major.
    {
      const __half* qrow = a.q + static_cast<int64_t>(row0 + qbase + (rv ? qi : 0)) * a.q_stride +
                           static_cast<int64_t>(g * a.group + hg) * D;
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {
        const int c = par * (D / 16) + cc;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rv) v = __ldg(reinterpret_cast<const uint4*>(qrow + c * 8));
        const uint32_t dst = q_s + (c >> 3) * C::kHalfBytes + swz128(r, c & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async();
      mbar_arrive(smem_addr(&q_full));
    }

    bool stopped = false;  // a wait of this thread gave up
    float m_run = -INFINITY, l_run = 0.f;
    const int min_pos = ctx + qbase;
    const bool prescale = !(a.scale_log2 > 0.f);
    const float mul = prescale ? 1.f : a.scale_log2;  // exponent = fma(score, mul, -m)
    for (int j = par; j < ntiles; j += 2) {
      const uint32_t sbuf = tmem + lane_addr + par * 128;
      // S_j done; it was issued after P_{j-2} V_{j-2}, so O_par is settled too.
      if (!mbar_wait(smem_addr(&s_full[par]), (j >> 1) & 1, a.err, a.wait_limit_ns)) {
        stopped = true;
        break;
      }
      tmem_fence_after_sync();
      uint32_t sv[C::kKeys / 32][32];
#pragma unroll
      for (int qq = 0; qq < C::kKeys / 32; ++qq) tmem_ld32(sbuf + qq * 32, sv[qq]);
      tmem_wait_ld();
#pragma unroll
      for (int qq = 0; qq < C::kKeys / 32; ++qq) tmem_regs_ready(sv[qq]);

      // Scores stay raw where scale > 0 (the max commutes with the scale, which is folded into
      // the exponent's FMA below); otherwise they are scaled here.  Masked keys become -inf.
      const int key0 = j * C::kKeys;
      const bool masked = !CASCADE && key0 + C::kKeys - 1 > min_pos;
      if (prescale || masked) {
#pragma unroll
        for (int c = 0; c < C::kKeys; ++c) {
          float v = __uint_as_float(sv[c >> 5][c & 31]);
          if (prescale) v *= a.scale_log2;
          if (masked && key0 + c > pos) v = -INFINITY;
          sv[c >> 5][c & 31] = __float_as_uint(v);
        }
      }
      float m2[2] = {-INFINITY, -INFINITY};  // two chains of three-input maxima
#pragma unroll
      for (int c = 0; c < C::kKeys; c += 2)
        m2[(c >> 1) & 1] = fmax3(m2[(c >> 1) & 1], __uint_as_float(sv[c >> 5][c & 31]),
                                 __uint_as_float(sv[c >> 5][(c & 31) + 1]));
      const float mx = fmaxf(m2[0], m2[1]) * mul;
      float alpha = 1.f;
      if (mx > m_run + C::kRescaleLog2 || (m_run == -INFINITY && mx > -INFINITY)) {
        alpha = ex2_approx(m_run - mx);  // 0 when m_run is still -inf
        m_run = mx;
      }
      if (j >= 2 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t t[32];
          tmem_ld32(obuf + c0, t);
          tmem_wait_ld();
          tmem_regs_ready(t);
#pragma unroll
          for (int c = 0; c < 32; ++c) t[c] = __float_as_uint(__uint_as_float(t[c]) * alpha);
          tmem_st32(obuf + c0, t);
        }
      }

      // P_j (fp16) -> TMEM columns 0..63 of the buffer, two keys per column; l keeps the
      // unrounded p.  A row with every key so far masked keeps m = -inf and gets p = 0.
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      // exponents and sums two keys at a time (packed fp32 pairs: the same roundings as fmaf
      // and + per key)
      const uint64_t mul2 = f32x2(mul, mul), negm2 = f32x2(neg_m, neg_m);
      uint64_t ps2[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
#pragma unroll
      for (int q8 = 0; q8 < C::kKeys / 16; ++q8) {  // 16 keys -> 8 columns of P at a time
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int k = q8 * 16 + 2 * c;
          float x0, x1;
          f32x2_split(ffma2(f32x2(__uint_as_float(sv[k >> 5][k & 31]),
                                  __uint_as_float(sv[k >> 5][(k & 31) + 1])),
                            mul2, negm2),
                      x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          ps2[c & 1] = fadd2(ps2[c & 1], f32x2(p0, p1));
          pk[c] = pack2<BF>(p0, p1);
        }
        tmem_st8(sbuf + q8 * 8, pk);
      }
      float s0, s1, s2, s3;
      f32x2_split(ps2[0], s0, s1);
      f32x2_split(ps2[1], s2, s3);
      l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));

      const int tile0 = j * C::kKeys;
      if (!CASCADE && j == ntiles - 1 && tile0 + C::kKeys > kend) {
        // The last tile: V rows at or past kend may be stale or NaN; zero them once the tile
        // has landed (the MMA reads V only after p_full below).  Thread r clears V row r.
        const int vst = j % C::kVStages;
        const bool landed = mbar_wait(smem_addr(&v_full[vst]), (j / C::kVStages) & 1,
                                      a.err, a.wait_limit_ns);
        if (landed && tile0 + r >= kend) {
          const uint32_t vrow = v_s + vst * C::kKVBytes + r * 128;
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               vrow + h * (C::kKeys * 128) + c * 16),
                           "r"(0u), "r"(0u), "r"(0u), "r"(0u)
                           : "memory");
        }
        fence_proxy_async();
        if (!landed) {
          stopped = true;
          break;
        }
      }
      tmem_wait_st();
      tmem_fence_before_sync();
      mbar_arrive(smem_addr(&p_full[par]));
    }

    // Merge the even and odd halves of each row: M = max, weights 2^(m - M).  The odd half
    // exists only when there are at least two key tiles.
    red_m[par][r] = m_run;
    red_l[par][r] = l_run;
    if (stopped) softmax_stop = 1;
    asm volatile("bar.sync 1, %0;" ::"n"(C::kSoftmax) : "memory");
    const bool two = ntiles >= 2;
    const float m_e = red_m[0][r], m_o = two ? red_m[1][r] : -INFINITY;
    const float mm = fmaxf(m_e, m_o);
    const float w_e = ex2_approx(m_e - mm), w_o = two ? ex2_approx(m_o - mm) : 0.f;
    const float l_all = red_l[0][r] * w_e + (two ? red_l[1][r] * w_o : 0.f);
    const float inv = a.v_scale / l_all;  // v_scale: 1, or the FP8 pool's V scale
    bool ok = !*reinterpret_cast<volatile int*>(&softmax_stop);
    if (ok) ok = mbar_wait(smem_addr(&drain), 0, a.err, a.wait_limit_ns);
    if (CASCADE && !__any_sync(0xffffffffu, !ok)) {
      // The rows' partials of the CTA's prefix partitions: m (log2 units), l, and this thread's
      // half of O / l.
      tmem_fence_after_sync();
      const int64_t pidx = (static_cast<int64_t>(qbase + qi) * a.num_q_heads + g * a.group + hg) *
                               a.max_parts + blockIdx.z * a.cascade_span;
      if (rv && par == 0) {
        a.part_m[pidx] = mm;
        a.part_l[pidx] = l_all;
      }
      const uint32_t oe = tmem + lane_addr + C::kOCol + par * kOHalf;
      float* dst = a.part_o + pidx * D + par * kOHalf;
#pragma unroll
      for (int c0 = 0; c0 < kOHalf; c0 += 32) {
        uint32_t te[32], to[32];
        tmem_ld32(oe + c0, te);
        tmem_ld32(oe + D + c0, to);
        tmem_wait_ld();
        tmem_regs_ready(te);
        tmem_regs_ready(to);
        if (rv) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dst + c0 + c) = make_float4(
                (__uint_as_float(te[c]) * w_e + __uint_as_float(to[c]) * w_o) * inv,
                (__uint_as_float(te[c + 1]) * w_e + __uint_as_float(to[c + 1]) * w_o) * inv,
                (__uint_as_float(te[c + 2]) * w_e + __uint_as_float(to[c + 2]) * w_o) * inv,
                (__uint_as_float(te[c + 3]) * w_e + __uint_as_float(to[c + 3]) * w_o) * inv);
        }
      }
    } else if (!CASCADE && !__any_sync(0xffffffffu, !ok)) {
      tmem_fence_after_sync();
      __half* dst = a.out + (static_cast<int64_t>(row0 + qbase + qi) * a.num_q_heads +
                             g * a.group + hg) * D + par * kOHalf;
      const uint32_t oe = tmem + lane_addr + C::kOCol + par * kOHalf;
#pragma unroll
      for (int c0 = 0; c0 < kOHalf; c0 += 32) {
        uint32_t te[32], to[32];
        tmem_ld32(oe + c0, te);
        if (two) tmem_ld32(oe + D + c0, to);
        tmem_wait_ld();
        tmem_regs_ready(te);
        if (two) tmem_regs_ready(to);
        auto o = [&](int c) {
          return (__uint_as_float(te[c]) * w_e + (two ? __uint_as_float(to[c]) * w_o : 0.f)) * inv;
        };
        if (rv) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 v;
            v.x = pack2<BF>(o(c), o(c + 1));
            v.y = pack2<BF>(o(c + 2), o(c + 3));
            v.z = pack2<BF>(o(c + 4), o(c + 5));
            v.w = pack2<BF>(o(c + 6), o(c + 7));
            *reinterpret_cast<uint4*>(dst + c0 + c) = v;
          }
        }
      }
    }
  }

  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
}

// Both kernels share the launch shape rules: 384 threads, one CTA per SM (TMEM and shared
// memory), and a register split that must fit the launch allocation.
template <typename C, typename K>
cudaError_t launch_one(K kern, const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       int q_tiles, cudaStream_t stream, bool cascade = false,
                       bool sliced = false) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc can only take registers the CTA was launched with: never launch a build
  // whose per-thread allocation is below the split (the increase would wait forever).
  cudaFuncAttributes attr{};
  if ((e = cudaFuncGetAttributes(&attr, kern)) != cudaSuccess) return e;
  if (attr.numRegs * C::kThreads < C::kRegsSoftmax * C::kSoftmax +
                                       C::kRegsOther * (C::kThreads - C::kSoftmax) ||
      attr.numRegs * C::kThreads > 65536)
    return cudaErrorInvalidConfiguration;
  // Query tokens per CTA: whole tokens per Q tile (128 / group rounds down), times the tiles.
  const int rows_q = q_tiles * (C::kRows / a.group);
  dim3 grid((a.max_query_len + rows_q - 1) / rows_q, a.num_kv_heads, a.prefill_seqs);
  if (!cascade && sliced && a.prefill_ctas > 0) {
    // A series of launches of prefill_ctas CTAs, each over the next slice of the items (heavy q
    // tiles of each chunk first): the prefill kernel then holds about that many SMs at a time,
    // and the decode kernel beside it (on another stream) gets the rest from the start.
    AttnArgs b = a;
    b.items_x = static_cast<int>(grid.x);
    const int64_t n_items = static_cast<int64_t>(grid.x) * grid.y * grid.z;
    for (int64_t base = 0; base < n_items; base += a.prefill_ctas) {
      b.item_base = static_cast<int>(base);
      const int n = static_cast<int>(std::min<int64_t>(a.prefill_ctas, n_items - base));
      kern<<<n, C::kThreads, C::kSmemBytes, stream>>>(kmap, vmap, b);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (cascade)  // every query row of the batch, every kv head, every group of prefix partitions
    grid = dim3(static_cast<unsigned>((a.num_tokens + rows_q - 1) / rows_q), a.num_kv_heads,
                a.cascade_parts / a.cascade_span);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

// Chunks that fit one Q tile (speculative verify, short chunks) go to the parity kernel, which
// splits their key tiles between two softmax warpgroups; longer chunks to the pair kernel,
// which gives each warpgroup its own Q tile and shares every K/V tile between them.
template <int D, int BS, bool BF, bool F8>
cudaError_t launch_prefill_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  if (a.max_query_len <= ParityCfg<D>::kRows / a.group)
    return launch_one<ParityCfg<D, F8>>(prefill_parity_kernel<D, BS, false, BF, F8>, a, kmap,
                                        vmap, 1, stream);
  return launch_one<PairCfg<D, F8>>(prefill_pair_kernel<D, BS, false, BF, F8>, a, kmap, vmap,
                                    PairCfg<D>::kQTiles, stream, false, true);
}

// The shared-prefix pass does 4 key tiles per CTA.  While the pair kernel's grid would leave
// SMs idle, one Q tile per CTA (the parity kernel: twice the CTAs, each key tile's softmax on
// its own warpgroup) finishes sooner; past that, the pair kernel's shared K/V tiles win.
template <int D, int BS, bool BF, bool F8>
cudaError_t launch_cascade_t(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  const int64_t rows_pair = PairCfg<D>::kQTiles * (PairCfg<D>::kRows / a.group);
  const int64_t pair_ctas = (a.num_tokens + rows_pair - 1) / rows_pair * a.num_kv_heads *
                            (a.cascade_parts / a.cascade_span);
  if (pair_ctas < a.num_sms)
    return launch_one<ParityCfg<D, F8>>(prefill_parity_kernel<D, BS, true, BF, F8>, a, kmap,
                                        vmap, 1, stream, true);
  return launch_one<PairCfg<D, F8>>(prefill_pair_kernel<D, BS, true, BF, F8>, a, kmap, vmap,
                                    PairCfg<D>::kQTiles, stream, true);
}

}  // namespace

namespace {

template <bool BF, bool F8>
cudaError_t launch_shared_prefix_b(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.block_size == 16 ? launch_cascade_t<128, 16, BF, F8>(a, kmap, vmap, stream)
                              : launch_cascade_t<128, 32, BF, F8>(a, kmap, vmap, stream);
  return a.block_size == 16 ? launch_cascade_t<64, 16, BF, F8>(a, kmap, vmap, stream)
                            : launch_cascade_t<64, 32, BF, F8>(a, kmap, vmap, stream);
}

template <bool BF, bool F8>
cudaError_t launch_prefill_b(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream) {
  if (a.head_dim == 128)
    return a.block_size == 16 ? launch_prefill_t<128, 16, BF, F8>(a, kmap, vmap, stream)
                              : launch_prefill_t<128, 32, BF, F8>(a, kmap, vmap, stream);
  return a.block_size == 16 ? launch_prefill_t<64, 16, BF, F8>(a, kmap, vmap, stream)
                            : launch_prefill_t<64, 32, BF, F8>(a, kmap, vmap, stream);
}

}  // namespace

cudaError_t launch_shared_prefix(const AttnArgs& a, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.kv_fp8) return launch_shared_prefix_b<false, true>(a, kmap, vmap, stream);
  return a.bf16 ? launch_shared_prefix_b<true, false>(a, kmap, vmap, stream)
                : launch_shared_prefix_b<false, false>(a, kmap, vmap, stream);
}

cudaError_t launch_prefill(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t stream) {
  if (a.kv_fp8) return launch_prefill_b<false, true>(a, kmap, vmap, stream);
  return a.bf16 ? launch_prefill_b<true, false>(a, kmap, vmap, stream)
                : launch_prefill_b<false, false>(a, kmap, vmap, stream);
}

}  // namespace pa
