// C ABI of the paged-attention library: argument checks, launch planning and status codes.
// See include/pa.h for the contract of every entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pa.h"
#include "pa_common.cuh"
#include "pa_kernels.h"

static_assert(PA_WAIT_LIMIT_DEFAULT_NS == pa::kWaitLimitNs, "default wait limit");

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_time_start[3] = {};  // indexed by PA_TIMED_*
thread_local cudaEvent_t g_time_stop[3] = {};
thread_local uint64_t g_wait_limit_ns = pa::kWaitLimitNs;  // pa_set_wait_limit

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// The device error word.  Kernels get its device address; pa_get_device_error reads it.
__device__ unsigned g_device_error_word;

constexpr int kMaxDevices = 256;
std::mutex g_err_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// Address of the error word on the current device (looked up once per device).
cudaError_t device_error_word(unsigned** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

// Error words of streams whose caller registered one (pa_set_stream_error_word): the kernels of
// a call on such a stream report into that word instead of the device's.  A few dozen entries,
// looked up under a mutex once per call.
constexpr int kMaxStreamWords = 64;
struct StreamWord {
  void* stream = nullptr;
  unsigned* word = nullptr;
};
std::mutex g_stream_mu;
StreamWord g_stream_words[kMaxStreamWords];

// The word a call on `stream` reports into: the stream's own, else the current device's.
cudaError_t error_word_for(void* stream, unsigned** out) {
  {
    std::lock_guard<std::mutex> lk(g_stream_mu);
    for (const StreamWord& w : g_stream_words)
      if (w.word && w.stream == stream) {
        *out = w.word;
        return cudaSuccess;
      }
  }
  return device_error_word(out);
}

// A side stream (highest priority) and two events per device and host thread: a call with both
// prefill chunks and decode rows runs the prefill kernel there, beside the decode and merge
// kernels on the caller's stream (fork and join through the events), so the HBM-bound decode
// grid fills the SMs the compute-bound prefill grid leaves idle in its tail.  Created on first
// use and kept for the thread's lifetime.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream g_side[kMaxDevices];

cudaError_t side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream& s = g_side[dev];
  if (!s.stream) {
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, greatest)) != cudaSuccess)
      return e;
  }
  *out = &s;
  return cudaSuccess;
}

// CTAs per launch of the two-tile prefill kernel beside the decode kernel (0: one full grid).
// The prefill launches hold whole SMs; the decode kernel streams on the rest.  When the decode
// rows carry at least about as much SM time as the prefill rows, the prefill goes as launches of
// two thirds of the SMs (the decode kernel keeps a third from the start); otherwise as one full
// grid.  The estimate: decode over prefill SM time ~ (decode rows / prefill rows) / G x 70 for
// contexts of similar length (one decode row moves Hkv d 4 bytes per key at ~75 GB/s per SM; one
// prefill row does 4 Hq d flops per key at ~5.3 TFLOP/s per SM), halved over an FP8 pool.
// Measured on the 4 x 512-row + 128-decode step (estimate 1.1; FP8 0.55), steps in us:
//   CTAs per launch    152    136    120    104    96     88     80     64     full grid
//   fp16 (bs 16)       447.6  454.2  441.6  424.5  425.3  431.0  562.9  493.9  458.9
//   FP8 pool           379.7                482.1         471.3  610.0  528.2  371.6
// Four or more launches in a row (80 CTAs and fewer here) chain the slowest CTA of each.  With
// 8 decode rows (estimate 0.07) one full grid takes 232.0 us against 275.0 in launches of 152.
int prefill_ctas_beside_decode(int num_sms, int64_t decode_rows, int64_t prefill_rows,
                               int group, bool fp8) {
  const double r = static_cast<double>(decode_rows) /
                   static_cast<double>(std::max<int64_t>(prefill_rows, 1)) / group * 70.0 *
                   (fp8 ? 0.5 : 1.0);
  return r >= 0.8 ? num_sms * 2 / 3 : 0;
}

// SM count of the current device (looked up once per device).
cudaError_t device_sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_sm_count[dev]) {
    e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  *out = g_sm_count[dev];
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool [NB, Hkv, bs, d] as a 2-D tensor of NB*Hkv*bs rows x d elements, in the layout the
// kernels' fragment loads expect.  fp16 / bf16: boxes of 16 rows x 64 values (128 bytes),
// 128-byte swizzle.  FP8: boxes of 16 rows x d bytes, 128-byte swizzle for d = 128 and none for
// d = 64 (a 64-byte row).
int make_pool_map(CUtensorMap* m, void* base, int64_t rows, int d, int dtype) {
  const bool fp8 = dtype == PA_F8E4M3;
  auto enc = tensor_map_encoder();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {fp8 ? static_cast<cuuint32_t>(d) : 64u, 16};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle swz =
      !fp8 || d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  const CUtensorMapDataType ty = fp8               ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = enc(m, ty, 2,
                   base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return PA_OK;
}

const char* dtype_name(int dt) {
  switch (dt) {
    case PA_F16: return "float16";
    case PA_I32: return "int32";
    case PA_I64: return "int64";
    case PA_F8E4M3: return "float8_e4m3";
    case PA_BF16: return "bfloat16";
    default: return "unknown";
  }
}

// Rank, dtype, non-negative shape, unit innermost stride, non-null data when non-empty.
int check_tensor(const pa_tensor* t, const char* name, int dtype, int ndim) {
  if (!t) return fail(PA_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (t->ndim != ndim)
    return fail(PA_ERR_INVALID_ARG, std::string(name) + " must have rank " + std::to_string(ndim) +
                                        ", got " + std::to_string(t->ndim));
  if (t->dtype != dtype)
    return fail(PA_ERR_INVALID_ARG, std::string(name) + " must be " + dtype_name(dtype) + ", got " +
                                        dtype_name(t->dtype));
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(PA_ERR_INVALID_ARG, std::string(name) + " has a negative dim");
    if (t->stride[i] < 0) return fail(PA_ERR_INVALID_ARG, std::string(name) + " has a negative stride");
    numel *= t->shape[i];
  }
  if (numel > 0) {
    if (!t->data) return fail(PA_ERR_INVALID_ARG, std::string(name) + " data is NULL");
    if (t->shape[ndim - 1] > 1 && t->stride[ndim - 1] != 1)
      return fail(PA_ERR_INVALID_ARG, std::string(name) + " innermost dim must be contiguous");
  }
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_contiguous(const pa_tensor* t, const char* name) {
  int64_t expect = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] > 1 && t->stride[i] != expect)
      return fail(PA_ERR_INVALID_ARG, std::string(name) + " must be contiguous");
    expect *= t->shape[i];
  }
  return PA_OK;
}

// Element type of a 16-bit pool entry point: bfloat16 when the pool says so, else fp16 (a pool
// of any other type then fails check_pool with a message naming float16).
int pool_dtype16(const pa_tensor* kc) { return kc && kc->dtype == PA_BF16 ? PA_BF16 : PA_F16; }

// Pool [NB, Hkv, bs, d] checks shared by both entry points.
int check_pool(const pa_tensor* kc, const pa_tensor* vc, int dtype = PA_F16) {
  int rc;
  if ((rc = check_tensor(kc, "k_cache", dtype, 4))) return rc;
  if ((rc = check_tensor(vc, "v_cache", dtype, 4))) return rc;
  for (int i = 0; i < 4; ++i)
    if (kc->shape[i] != vc->shape[i])
      return fail(PA_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  if ((rc = check_contiguous(kc, "k_cache"))) return rc;
  if ((rc = check_contiguous(vc, "v_cache"))) return rc;
  const int64_t d = kc->shape[3], bs = kc->shape[2];
  if (d != 64 && d != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim " + std::to_string(d) + " not built (64, 128)");
  if (bs != 16 && bs != 32)
    return fail(PA_ERR_UNSUPPORTED, "block_size " + std::to_string(bs) + " not built (16, 32)");
  if (kc->shape[1] < 1 || kc->shape[1] > 65535)
    return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be in 1..65535");
  if (kc->shape[0] * kc->shape[1] * bs >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "pool has 2^31 or more token rows");
  if (kc->shape[0] > 0 && (!aligned16(kc->data) || !aligned16(vc->data)))
    return fail(PA_ERR_INVALID_ARG, "k_cache / v_cache must be 16-byte aligned");
  return PA_OK;
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WorkspaceLayout {
  size_t o_bytes, m_off, l_off, total;
};

WorkspaceLayout workspace_layout(int64_t t, int64_t hq, int64_t d, int32_t max_seq_len) {
  WorkspaceLayout w{0, 0, 0, 0};
  const int64_t parts = max_seq_len > 0 ? (max_seq_len + PA_PARTITION_TOKENS - 1) / PA_PARTITION_TOKENS : 0;
  if (parts <= 1 || t <= 0) return w;
  const size_t rows = static_cast<size_t>(t) * hq * parts;
  w.o_bytes = align_up(rows * d * sizeof(float), 256);
  w.m_off = w.o_bytes;
  w.l_off = w.m_off + align_up(rows * sizeof(float), 256);
  w.total = w.l_off + align_up(rows * sizeof(float), 256);
  return w;
}

}  // namespace

namespace pa {
int set_last_error(int status, const std::string& message) { return fail(status, message); }
cudaError_t error_word(void* stream, unsigned** out) { return error_word_for(stream, out); }
}  // namespace pa

extern "C" {

const char* pa_last_error(void) { return g_last_error.c_str(); }

int pa_version(void) { return PA_VERSION; }

size_t pa_attention_workspace_size(int64_t num_tokens, int64_t num_q_heads, int64_t head_dim,
                                   int32_t max_seq_len) {
  return workspace_layout(num_tokens, num_q_heads, head_dim, max_seq_len).total;
}

static int check_scales(const pa_kv_scales* sc) {
  if (!sc) return fail(PA_ERR_INVALID_ARG, "scales is NULL");
  for (float x : {sc->k_scale, sc->v_scale})
    if (!(x > 0.f) || !(x < INFINITY))
      return fail(PA_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
  return PA_OK;
}

// The scatter-write into an fp16 cache (sc == NULL) or an FP8 cache with scales sc.
static int reshape_impl(const pa_tensor* k, const pa_tensor* v, const pa_tensor* k_cache,
                        const pa_tensor* v_cache, const pa_tensor* slot_mapping,
                        const pa_kv_scales* sc, bool fp8, void* stream) {
  g_last_error.clear();
  int rc;
  if (fp8 && (rc = check_scales(sc))) return rc;
  // fp16 or bf16 tokens into a pool of the same type; fp16 tokens into an FP8 pool
  const int in_dt = fp8 ? PA_F16 : pool_dtype16(k_cache);
  if ((rc = check_pool(k_cache, v_cache, fp8 ? PA_F8E4M3 : in_dt))) return rc;
  if ((rc = check_tensor(k, "k", in_dt, 3))) return rc;
  if ((rc = check_tensor(v, "v", in_dt, 3))) return rc;
  if ((rc = check_tensor(slot_mapping, "slot_mapping", PA_I64, 1))) return rc;
  const int64_t t = k->shape[0], hkv = k_cache->shape[1], d = k_cache->shape[3];
  for (const pa_tensor* x : {k, v}) {
    if (x->shape[0] != t || x->shape[1] != hkv || x->shape[2] != d)
      return fail(PA_ERR_INVALID_ARG, "k and v must be [T_new, num_kv_heads, head_dim] matching the pool");
    if (t > 0 && ((x->shape[1] > 1 && x->stride[1] != d) || x->stride[0] < hkv * d ||
                  x->stride[0] % 8 != 0 || !aligned16(x->data)))
      return fail(PA_ERR_INVALID_ARG,
                  "k / v need head stride head_dim, token stride >= heads*head_dim and a multiple "
                  "of 8, and 16-byte alignment");
  }
  if (slot_mapping->shape[0] != t)
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must have T_new entries");
  if (t == 0) return PA_OK;

  pa::CacheArgs a{};
  a.k = static_cast<const __half*>(k->data);
  a.v = static_cast<const __half*>(v->data);
  a.k_stride = k->stride[0];
  a.v_stride = v->stride[0];
  a.k_cache = k_cache->data;
  a.v_cache = v_cache->data;
  a.fp8 = fp8 ? 1 : 0;
  a.k_inv = fp8 ? 1.0f / sc->k_scale : 1.f;
  a.v_inv = fp8 ? 1.0f / sc->v_scale : 1.f;
  a.slot_mapping = static_cast<const int64_t*>(slot_mapping->data);
  a.num_tokens = t;
  a.num_kv_heads = static_cast<int>(hkv);
  a.head_dim = static_cast<int>(d);
  a.block_size = static_cast<int>(k_cache->shape[2]);
  a.num_blocks = k_cache->shape[0];
  cudaError_t e = error_word_for(stream, &a.err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  e = pa::launch_reshape_and_cache(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  return PA_OK;
}

int pa_reshape_and_cache(const pa_tensor* k, const pa_tensor* v, const pa_tensor* k_cache,
                         const pa_tensor* v_cache, const pa_tensor* slot_mapping, void* stream) {
  return reshape_impl(k, v, k_cache, v_cache, slot_mapping, nullptr, false, stream);
}

int pa_reshape_and_cache_fp8(const pa_tensor* k, const pa_tensor* v, const pa_tensor* k_cache,
                             const pa_tensor* v_cache, const pa_tensor* slot_mapping,
                             const pa_kv_scales* scales, void* stream) {
  return reshape_impl(k, v, k_cache, v_cache, slot_mapping, scales, true, stream);
}

int pa_copy_blocks(const pa_tensor* k_cache, const pa_tensor* v_cache, const pa_tensor* pairs,
                   void* stream) {
  g_last_error.clear();
  int rc;
  const bool fp8 = k_cache && k_cache->dtype == PA_F8E4M3;
  if ((rc = check_pool(k_cache, v_cache, fp8 ? PA_F8E4M3 : pool_dtype16(k_cache)))) return rc;
  if ((rc = check_tensor(pairs, "pairs", PA_I32, 2))) return rc;
  if (pairs->shape[1] != 2 || (pairs->shape[0] > 1 && pairs->stride[0] != 2))
    return fail(PA_ERR_INVALID_ARG, "pairs must be a contiguous int32 [n, 2] array");
  if (pairs->shape[0] == 0) return PA_OK;
  pa::CopyArgs a{};
  a.k_cache = static_cast<uint4*>(k_cache->data);
  a.v_cache = static_cast<uint4*>(v_cache->data);
  a.pairs = static_cast<const int32_t*>(pairs->data);
  a.num_pairs = pairs->shape[0];
  a.chunks_per_block = k_cache->shape[1] * k_cache->shape[2] * k_cache->shape[3] / (fp8 ? 16 : 8);
  a.num_blocks = k_cache->shape[0];
  cudaError_t e = error_word_for(stream, &a.err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  e = pa::launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PA_OK;
}

// Attention over an fp16 cache (fp8 false) or an FP8 cache with scales sc.
static int attention_impl(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                          const pa_tensor* block_tables, const pa_tensor* seq_lens,
                          const pa_tensor* query_start_loc, float scale, const pa_tensor* out,
                          const pa_batch_hint* hint, const pa_kv_scales* sc, bool fp8,
                          void* workspace, size_t workspace_bytes, void* stream) {
  g_last_error.clear();
  int rc;
  if (fp8 && (rc = check_scales(sc))) return rc;
  // q, out and the pools all fp16 or all bf16; fp16 q and out over an FP8 pool
  const int in_dt = fp8 ? PA_F16 : pool_dtype16(k_cache);
  if ((rc = check_pool(k_cache, v_cache, fp8 ? PA_F8E4M3 : in_dt))) return rc;
  if ((rc = check_tensor(q, "q", in_dt, 3))) return rc;
  if ((rc = check_tensor(out, "out", in_dt, 3))) return rc;
  if ((rc = check_tensor(block_tables, "block_tables", PA_I32, 2))) return rc;
  if ((rc = check_tensor(seq_lens, "seq_lens", PA_I32, 1))) return rc;
  if ((rc = check_tensor(query_start_loc, "query_start_loc", PA_I32, 1))) return rc;
  if (!hint) return fail(PA_ERR_INVALID_ARG, "hint is NULL");
  const int64_t t = q->shape[0], hq = q->shape[1], d = q->shape[2];
  const int64_t hkv = k_cache->shape[1];
  const int64_t n = seq_lens->shape[0];
  if (d != k_cache->shape[3]) return fail(PA_ERR_INVALID_ARG, "q head_dim differs from the pool's");
  if (hq < 1 || hq % hkv != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
  const int64_t group = hq / hkv;
  if (group > 16) return fail(PA_ERR_UNSUPPORTED, "GQA group size above 16 not built");
  if (out->shape[0] != t || out->shape[1] != hq || out->shape[2] != d)
    return fail(PA_ERR_INVALID_ARG, "out must be [T, num_q_heads, head_dim] like q");
  if ((rc = check_contiguous(out, "out"))) return rc;
  if (t > 0 && ((hq > 1 && q->stride[1] != d) || q->stride[0] < hq * d || q->stride[0] % 8 != 0 ||
                !aligned16(q->data) || !aligned16(out->data)))
    return fail(PA_ERR_INVALID_ARG,
                "q needs head stride head_dim, token stride >= heads*head_dim and a multiple of 8; "
                "q and out need 16-byte alignment");
  if (query_start_loc->shape[0] != n + 1)
    return fail(PA_ERR_INVALID_ARG, "query_start_loc must have num_seqs + 1 entries");
  if (block_tables->shape[0] != n)
    return fail(PA_ERR_INVALID_ARG, "block_tables must have num_seqs rows");
  if (n > 65535) return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences in one call");
  if (block_tables->shape[1] < 1 && n > 0)
    return fail(PA_ERR_INVALID_ARG, "block_tables needs at least one column");
  if (block_tables->shape[1] > INT32_MAX || block_tables->stride[0] < block_tables->shape[1])
    return fail(PA_ERR_INVALID_ARG, "block_tables row stride must cover its columns");
  if (hint->max_query_len < 0 || hint->max_seq_len < 0 || hint->num_prefill_seqs < 0 ||
      hint->shared_prefix_tokens < 0)
    return fail(PA_ERR_INVALID_ARG, "hint values must be non-negative");
  const int64_t bs = k_cache->shape[2];
  const int sp = hint->shared_prefix_tokens;
  if (sp > 0) {
    if (sp % PA_PARTITION_TOKENS != 0 || sp % bs != 0)
      return fail(PA_ERR_INVALID_ARG, "shared_prefix_tokens must be a multiple of 512 and of the "
                                      "block size");
    if (sp >= hint->max_seq_len || sp / bs > block_tables->shape[1])
      return fail(PA_ERR_INVALID_ARG, "shared_prefix_tokens must be below max_seq_len and within "
                                      "the block tables");
    if (hint->max_query_len > 1)
      return fail(PA_ERR_UNSUPPORTED, "the shared-prefix pass is built for decode rows");
  }
  if (hint->max_query_len > hint->max_seq_len)
    return fail(PA_ERR_INVALID_ARG, "hint max_query_len exceeds max_seq_len");
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN");
  // Verify rows: when every sequence has at most a few query rows, the decode kernel can serve
  // them all, each column (query row, head) with its own causal limit: one read of a 512-key
  // partition feeds every column, and no prefill launch is made.  It does so for up to 8
  // columns (where a 128-row prefill tile would be mostly empty), and over an FP8 cache (which
  // the prefill kernels do not read) for up to 32.  Between 8 and 32 columns over fp16/bf16 the
  // key-parity prefill kernel is as fast and needs no merge.
  const int64_t group_size = hq % hkv == 0 && hkv > 0 ? hq / hkv : 1;
  const int64_t verify_cols = hint->max_query_len * group_size;
  const bool verify = hint->max_query_len > 1 && (verify_cols <= 8 || (fp8 && verify_cols <= 32));

  const WorkspaceLayout ws = workspace_layout(t, hq, d, hint->max_seq_len);
  if (ws.total > 0) {
    if (!workspace || workspace_bytes < ws.total)
      return fail(PA_ERR_WORKSPACE, "workspace needs " + std::to_string(ws.total) + " bytes");
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(PA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  }
  if (t == 0 || n == 0 || hint->max_query_len == 0) return PA_OK;

  pa::AttnArgs a{};
  a.q = static_cast<const __half*>(q->data);
  a.q_stride = q->stride[0];
  a.out = static_cast<__half*>(out->data);
  a.block_tables = static_cast<const int32_t*>(block_tables->data);
  a.bt_stride = block_tables->stride[0];
  a.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  a.query_start_loc = static_cast<const int32_t*>(query_start_loc->data);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  a.part_o = ws.total ? reinterpret_cast<float*>(wsb) : nullptr;
  a.part_m = ws.total ? reinterpret_cast<float*>(wsb + ws.m_off) : nullptr;
  a.part_l = ws.total ? reinterpret_cast<float*>(wsb + ws.l_off) : nullptr;
  a.num_seqs = static_cast<int>(n);
  a.num_tokens = t;
  a.num_q_heads = static_cast<int>(hq);
  a.num_kv_heads = static_cast<int>(hkv);
  a.group = static_cast<int>(group);
  a.head_dim = static_cast<int>(d);
  a.block_size = static_cast<int>(k_cache->shape[2]);
  a.max_blocks = static_cast<int>(block_tables->shape[1]);
  a.num_blocks = k_cache->shape[0];
  a.max_parts = static_cast<int>(
      std::max<int64_t>(1, (hint->max_seq_len + PA_PARTITION_TOKENS - 1) / PA_PARTITION_TOKENS));
  a.max_query_len = hint->max_query_len;
  a.prefill_seqs = hint->num_prefill_seqs > 0 ? std::min<int>(hint->num_prefill_seqs, n) : n;
  // Every sequence has several rows (by the hint) and the prefill kernel serves them: no decode
  // rows, so no decode or merge launch.
  const bool all_prefill = !verify && hint->max_query_len > 1 && hint->num_prefill_seqs >= n;
  a.decode_skipped = all_prefill ? 1 : 0;
  a.verify_rows = verify ? hint->max_query_len : 1;
  const int cols_per_cta = group * a.verify_rows <= 8 ? 8 : 16;
  a.col_groups = static_cast<int>((group * a.verify_rows + cols_per_cta - 1) / cols_per_cta);
  // FP8: K = k_scale * code value, so the score scale takes k_scale; V's scale goes on the output.
  a.scale_log2 = scale * 1.4426950408889634f * (fp8 ? sc->k_scale : 1.f);
  a.v_scale = fp8 ? sc->v_scale : 1.f;
  a.kv_fp8 = fp8 ? 1 : 0;
  a.bf16 = in_dt == PA_BF16 ? 1 : 0;
  a.cascade_parts = sp / PA_PARTITION_TOKENS;
  // The shared-prefix pass runs beside the decode kernel on the side stream, each CTA over two
  // prefix partitions when their number is even (one otherwise).  Measured on 160 rows behind a
  // 2048-key prefix (step, us): after the decode kernel as its programmatic dependent 61.1 (two
  // partitions per CTA 64.0, four 70.8); beside it 66.0 / 59.1 / 62.5 for one / two / four; over
  // an FP8 pool 52.4 after it, 52.6 beside it with two.
  a.cascade_span = a.cascade_parts % 2 == 0 ? 2 : 1;
  a.wait_limit_ns = g_wait_limit_ns;
  cudaError_t e = error_word_for(stream, &a.err);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  if (a.cascade_parts > 0 && (e = device_sm_count(&a.num_sms)) != cudaSuccess)
    return cuda_fail(e, "device attribute");

  const int64_t rows = k_cache->shape[0] * hkv * k_cache->shape[2];
  CUtensorMap kmap, vmap;
  const int pool_dt = k_cache->dtype;
  if ((rc = make_pool_map(&kmap, k_cache->data, rows, static_cast<int>(d), pool_dt))) return rc;
  if ((rc = make_pool_map(&vmap, v_cache->data, rows, static_cast<int>(d), pool_dt))) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto mark = [&](int kernel, bool stop, cudaStream_t on) {
    cudaEvent_t ev = stop ? g_time_stop[kernel] : g_time_start[kernel];
    return ev ? cudaEventRecord(ev, on) : cudaSuccess;
  };
  auto prefill = [&](cudaStream_t on) -> int {
    cudaError_t err;
    if ((err = mark(PA_TIMED_PREFILL, false, on)) != cudaSuccess) return cuda_fail(err, "timing event");
    if ((err = pa::launch_prefill(a, kmap, vmap, on)) != cudaSuccess)
      return cuda_fail(err, "prefill launch");
    if ((err = mark(PA_TIMED_PREFILL, true, on)) != cudaSuccess) return cuda_fail(err, "timing event");
    return PA_OK;
  };
  // Prefill chunks next to decode rows, or the shared-prefix pass: it goes first, on the side
  // stream, and the caller's stream waits for it (the join): for prefill chunks after its own
  // launches, for the pass before the merge that reads its partials; on every return path.
  struct Join {
    SideStream* side = nullptr;
    cudaStream_t st = nullptr;
    cudaError_t done() {
      if (!side) return cudaSuccess;
      cudaError_t je = cudaEventRecord(side->join, side->stream);
      if (je == cudaSuccess) je = cudaStreamWaitEvent(st, side->join, 0);
      side = nullptr;
      return je;
    }
    ~Join() { done(); }
  } join;
  if (!all_prefill && !verify && hint->max_query_len > 1) {
    if ((e = device_sm_count(&a.num_sms)) != cudaSuccess) return cuda_fail(e, "device attribute");
    const int64_t decode_rows = n - a.prefill_seqs;
    a.prefill_ctas = prefill_ctas_beside_decode(a.num_sms, decode_rows, t - decode_rows, a.group,
                                                fp8);
    SideStream* side = nullptr;
    if ((e = side_stream(&side)) != cudaSuccess) return cuda_fail(e, "side stream");
    if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess)
      return cuda_fail(e, "stream fork");
    join.side = side;
    join.st = st;
    if ((rc = prefill(side->stream))) return rc;
  }
  auto mark_st = [&](int kernel, bool stop) { return mark(kernel, stop, st); };
  if (a.cascade_parts > 0) {  // the pass first, on the side stream; the merge waits for it
    SideStream* side = nullptr;
    if ((e = side_stream(&side)) != cudaSuccess) return cuda_fail(e, "side stream");
    if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess)
      return cuda_fail(e, "stream fork");
    join.side = side;
    join.st = st;
    if ((e = mark(PA_TIMED_SHARED_PREFIX, false, side->stream)) != cudaSuccess)
      return cuda_fail(e, "timing event");
    e = pa::launch_shared_prefix(a, kmap, vmap, side->stream);
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix launch");
    if ((e = mark(PA_TIMED_SHARED_PREFIX, true, side->stream)) != cudaSuccess)
      return cuda_fail(e, "timing event");
  }
  if (!all_prefill) {
    if ((e = mark_st(PA_TIMED_DECODE, false)) != cudaSuccess) return cuda_fail(e, "timing event");
    e = pa::launch_decode(a, kmap, vmap, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    if ((e = mark_st(PA_TIMED_DECODE, true)) != cudaSuccess) return cuda_fail(e, "timing event");
  }
  if (a.cascade_parts > 0 && (e = join.done()) != cudaSuccess) return cuda_fail(e, "stream join");
  if (a.max_parts > 1 && !all_prefill) {
    e = pa::launch_merge(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  if (all_prefill) return prefill(st);  // only prefill chunks: everything on the caller's stream
  if ((e = join.done()) != cudaSuccess) return cuda_fail(e, "stream join");
  return PA_OK;
}

int pa_attention(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* block_tables, const pa_tensor* seq_lens,
                 const pa_tensor* query_start_loc, float scale, const pa_tensor* out,
                 const pa_batch_hint* hint, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return attention_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                        hint, nullptr, false, workspace, workspace_bytes, stream);
}

int pa_attention_fp8(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                     const pa_tensor* block_tables, const pa_tensor* seq_lens,
                     const pa_tensor* query_start_loc, float scale, const pa_tensor* out,
                     const pa_batch_hint* hint, const pa_kv_scales* scales, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return attention_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                        hint, scales, true, workspace, workspace_bytes, stream);
}

int pa_set_timing_events(int kernel, void* start, void* stop) {
  g_last_error.clear();
  if (kernel != PA_TIMED_DECODE && kernel != PA_TIMED_PREFILL && kernel != PA_TIMED_SHARED_PREFIX)
    return fail(PA_ERR_INVALID_ARG,
                "timed kernel must be PA_TIMED_DECODE, PA_TIMED_PREFILL or PA_TIMED_SHARED_PREFIX");
  const bool on = start && stop;
  g_time_start[kernel] = on ? static_cast<cudaEvent_t>(start) : nullptr;
  g_time_stop[kernel] = on ? static_cast<cudaEvent_t>(stop) : nullptr;
  return PA_OK;
}

int pa_set_wait_limit(uint64_t limit_ns) {
  g_last_error.clear();
  if (limit_ns < PA_WAIT_LIMIT_MIN_NS || limit_ns > PA_WAIT_LIMIT_MAX_NS)
    return fail(PA_ERR_INVALID_ARG, "wait limit must be in [" +
                                        std::to_string(PA_WAIT_LIMIT_MIN_NS) + ", " +
                                        std::to_string(PA_WAIT_LIMIT_MAX_NS) + "] ns");
  g_wait_limit_ns = limit_ns;
  return PA_OK;
}

int pa_set_stream_error_word(void* stream, uint32_t* device_word) {
  g_last_error.clear();
  if (device_word && (reinterpret_cast<uintptr_t>(device_word) & 3u))
    return fail(PA_ERR_INVALID_ARG, "the error word must be 4-byte aligned");
  std::lock_guard<std::mutex> lk(g_stream_mu);
  StreamWord* slot = nullptr;
  for (StreamWord& w : g_stream_words)
    if (w.word && w.stream == stream) slot = &w;
  if (!device_word) {  // back to the device's word
    if (slot) *slot = StreamWord{};
    return PA_OK;
  }
  if (!slot)
    for (StreamWord& w : g_stream_words)
      if (!w.word) {
        slot = &w;
        break;
      }
  if (!slot)
    return fail(PA_ERR_INVALID_ARG, "already " + std::to_string(kMaxStreamWords) +
                                        " streams hold an error word of their own");
  slot->stream = stream;
  slot->word = reinterpret_cast<unsigned*>(device_word);
  return PA_OK;
}

int pa_get_device_error(void* stream, uint32_t* bits) {
  g_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned* p = nullptr;
  e = error_word_for(stream, &p);
  if (e != cudaSuccess) return cuda_fail(e, "error word");
  unsigned w = 0;
  e = cudaMemcpy(&w, p, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const unsigned zero = 0;
  e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  if (bits) *bits = w;
  if (w & pa::kErrTimeout) return fail(PA_ERR_TIMEOUT, "a device wait timed out");
  if (w & (pa::kErrSlotRange | pa::kErrBlockRange))
    return fail(PA_ERR_OUT_OF_RANGE, "a slot or block id outside the pool was skipped");
  if (w & (pa::kErrDescriptor | pa::kErrHint))
    return fail(PA_ERR_DESCRIPTOR, "a sequence's descriptor was invalid or exceeded the hint");
  return PA_OK;
}

}  // extern "C"
