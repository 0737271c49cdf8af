// Host side of the C ABI (include/cpattn.h): argument validation, error reporting and the
// launches of the integer layout kernels and the LSE merge.  Attention kernels live in
// prefill_tc.cu, prefill_simt.cu and decode.cu.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"

namespace {

thread_local char g_detail[512] = "";
thread_local int32_t g_status = CP_OK;

cp_status fail(cp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  g_status = st;
  return st;
}

cp_status ok() {
  g_status = CP_OK;
  g_detail[0] = '\0';
  return CP_OK;
}

cp_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(CP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return ok();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, ...)                                   \
  do {                                                       \
    if (!(cond)) return fail(CP_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define REQUIRE_PTR(p) REQUIRE((p) != nullptr && aligned16(p), #p " must be a non-null 16-byte aligned pointer")

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

// ============================================================================ device kernels
namespace cpattn {
namespace {

// ---- cp_partition: per-(rank, sequence) row offsets in shared memory, then one thread per
// token.  Offsets: off[r][b] = rows of rank r that precede sequence b, base[r] = rows of the
// ranks before r.
__global__ void partition_kernel(const int32_t* __restrict__ cu, int B, int N, int cp,
                                 int32_t* perm, int32_t* inv, int32_t* shard_offsets,
                                 int32_t* chunk_bounds) {
  extern __shared__ int32_t sm[];
  int32_t* off = sm;                  // [cp][B + 1]
  int32_t* base = sm + cp * (B + 1);  // [cp + 1]
  for (int i = threadIdx.x; i < cp * B; i += blockDim.x) {
    const int r = i / B, b = i % B;
    const int T = cu[b + 1] - cu[b];
    const int c2 = 2 * cp - 1 - r;
    off[r * (B + 1) + b + 1] = (chunk_bound(r + 1, T, cp) - chunk_bound(r, T, cp)) +
                               (chunk_bound(c2 + 1, T, cp) - chunk_bound(c2, T, cp));
  }
  __syncthreads();
  for (int r = threadIdx.x; r < cp; r += blockDim.x) {
    int32_t* o = off + r * (B + 1);
    o[0] = 0;
    for (int b = 0; b < B; ++b) o[b + 1] += o[b];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    base[0] = 0;
    for (int r = 0; r < cp; ++r) base[r + 1] = base[r] + off[r * (B + 1) + B];
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    if (shard_offsets)
      for (int r = threadIdx.x; r <= cp; r += blockDim.x) shard_offsets[r] = base[r];
    if (chunk_bounds)
      for (int i = threadIdx.x; i < B * (2 * cp + 1); i += blockDim.x) {
        const int b = i / (2 * cp + 1), k = i % (2 * cp + 1);
        chunk_bounds[i] = chunk_bound(k, cu[b + 1] - cu[b], cp);
      }
  }
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < N; t += gridDim.x * blockDim.x) {
    const int b = seq_of_row(cu, B, t);
    const int T = cu[b + 1] - cu[b];
    const int o = t - cu[b];
    const int c = chunk_of(o, T, cp);
    const int r = shard_of_chunk(c, cp);
    const int within = (c == r) ? o - chunk_bound(r, T, cp)
                                : (chunk_bound(r + 1, T, cp) - chunk_bound(r, T, cp)) +
                                      (o - chunk_bound(c, T, cp));
    const int row = base[r] + off[r * (B + 1) + b] + within;
    if (row >= N) continue;  // total_tokens smaller than cu_seqlens[B]: caller error, no write
    if (perm) perm[row] = t;
    if (inv) inv[t] = row;
  }
}

// ---- cp_kv_interleave_layout: closed forms of the round-robin deal, one thread per item.
__global__ void interleave_kernel(const int32_t* __restrict__ cu, int B, int N, int cp, int I,
                                  int bs, const int32_t* __restrict__ tables, int max_blocks,
                                  int32_t* local_lens, int32_t* rank_of, int32_t* local_of,
                                  int64_t* slot_of, int32_t* err) {
  const long long items = max((long long)N, (long long)cp * B);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < items;
       i += (long long)gridDim.x * blockDim.x) {
    if (local_lens && i < (long long)cp * B) {
      const int r = (int)(i / B), b = (int)(i % B);
      local_lens[i] = rank_local_len(cu[b + 1] - cu[b], r, cp, I);
    }
    if (i < N) {
      const int t = (int)i;
      const int b = seq_of_row(cu, B, t);
      const long long p = t - cu[b];
      const int r = (int)((p / I) % cp);
      const long long l = (p / ((long long)I * cp)) * I + p % I;
      if (rank_of) rank_of[t] = r;
      if (local_of) local_of[t] = (int32_t)l;
      if (slot_of) {
        const long long col = l / bs;
        long long slot = -1;
        if (col < max_blocks) {
          const int page = tables[((long long)r * B + b) * max_blocks + col];
          if (page >= 0) slot = (long long)page * bs + l % bs;
        }
        if (slot < 0) report(err, CP_ERR_DEVICE_BOUNDS);
        slot_of[t] = slot;
      }
    }
  }
}

// ---- cp_kv_cache_write: one thread per 16-byte vector of a new token's K and V rows.
__global__ void kv_write_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                const int32_t* __restrict__ cu, const int32_t* __restrict__ start,
                                int B, int N, int Hkv, int vecs, int cp, int I, int bs,
                                const int32_t* __restrict__ tables, int max_blocks,
                                long long pool, uint4* k_cache, uint4* v_cache, int32_t* err) {
  const long long total = (long long)N * Hkv * vecs;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int vec = (int)(i % vecs);
    const int g = (int)((i / vecs) % Hkv);
    const int t = (int)(i / ((long long)vecs * Hkv));
    const int b = seq_of_row(cu, B, t);
    const long long pos = (long long)start[b] + (t - cu[b]);
    const int r = (int)((pos / I) % cp);
    const long long l = (pos / ((long long)I * cp)) * I + pos % I;
    const long long col = l / bs;
    const int page = col < max_blocks ? tables[((long long)r * B + b) * max_blocks + col] : -1;
    if (page < 0 || page >= pool) {
      report(err, CP_ERR_DEVICE_BOUNDS);
      continue;
    }
    const long long dst = ((((long long)r * pool + page) * Hkv + g) * bs + l % bs) * vecs + vec;
    k_cache[dst] = k_new[i];
    v_cache[dst] = v_new[i];
  }
}

// ---- cp_lse_merge: one warp per (row, head); lanes own D/32 consecutive floats.
template <int D>
struct MergeVec;
template <>
struct MergeVec<128> {
  using T = float4;
  static CP_DEV void fma(float (&acc)[4], float w, const T& x) {
    acc[0] += w * x.x;
    acc[1] += w * x.y;
    acc[2] += w * x.z;
    acc[3] += w * x.w;
  }
};
template <>
struct MergeVec<64> {
  using T = float2;
  static CP_DEV void fma(float (&acc)[2], float w, const T& x) {
    acc[0] += w * x.x;
    acc[1] += w * x.y;
  }
};

template <int D, bool BF16_OUT>
CP_DEV void merge_store(void* out, float* out_lse, long long u, int lane, const float (&acc)[D / 32],
                        float wsum, float M) {
  constexpr int E = D / 32;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  if constexpr (BF16_OUT) {
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + u * D + lane * E;
    if constexpr (E == 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&a);
      pk.y = *reinterpret_cast<uint32_t*>(&b);
      *reinterpret_cast<uint2*>(o) = pk;
    } else {
      *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    }
  } else {
    float* o = static_cast<float*>(out) + u * D + lane * E;
    if constexpr (E == 4) {
      *reinterpret_cast<float4*>(o) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
      *reinterpret_cast<float2*>(o) = make_float2(acc[0] * inv, acc[1] * inv);
    }
  }
  if (out_lse && lane == 0) out_lse[u] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

// Few partials (the prefill case): the P LSEs of a unit are loaded together, then the rows of
// the non-empty partials together (an empty partial's row is never read: in causal prefill
// about one row in eight is empty, and measured, skipping those reads beats issuing every
// load in one round trip).
// (row, head) units per warp in merge_small_kernel: 2 measured best (1: 4 µs slower on the
// full prefill's merge, 4: 2 µs slower)
constexpr int kMergeUnits = 2;

template <int D, bool BF16_OUT, int P>
__global__ void __launch_bounds__(256) merge_small_kernel(const float* __restrict__ po,
                                                          const float* __restrict__ pl,
                                                          long long units, void* out,
                                                          float* out_lse) {
  constexpr int E = D / 32, U = kMergeUnits;
  using V = typename MergeVec<D>::T;
  griddep_wait();  // the partials' producer may still be finishing
  // U units per warp, every load of all of them issued before any arithmetic (twice the
  // bytes in flight of one unit per warp)
  const long long u0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * U;
  const int lane = threadIdx.x & 31;
  if (u0 >= units) return;
  float lp[U][P];
  V x[U][P];
#pragma unroll
  for (int j = 0; j < U; ++j)
#pragma unroll
    for (int p = 0; p < P; ++p)
      lp[j][p] = u0 + j < units ? __ldg(pl + (long long)p * units + u0 + j) * kLog2e : -INFINITY;
#pragma unroll
  for (int j = 0; j < U; ++j)
#pragma unroll
    for (int p = 0; p < P; ++p) {
      if (lp[j][p] > -INFINITY)
        x[j][p] = __ldg(reinterpret_cast<const V*>(po + ((long long)p * units + u0 + j) * D + lane * E));
      else
        x[j][p] = V{};
    }
#pragma unroll
  for (int j = 0; j < U; ++j) {
    if (u0 + j >= units) break;
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < P; ++p) M = fmaxf(M, lp[j][p]);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int p = 0; p < P; ++p) {
        const bool live = lp[j][p] > -INFINITY;
        const float w = live ? exp2f(lp[j][p] - M) : 0.f;
        wsum += w;
        if (live) MergeVec<D>::fma(acc, w, x[j][p]);
      }
    }
    merge_store<D, BF16_OUT>(out, out_lse, u0 + j, lane, acc, wsum, M);
  }
}

// Any number of partials (the decode case, cp x splits): LSEs read 32 at a time across the
// lanes; only non-empty partials' rows are read.
template <int D, bool BF16_OUT>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ po,
                                                    const float* __restrict__ pl, int P,
                                                    long long units, void* out, float* out_lse) {
  constexpr int E = D / 32;
  using V = typename MergeVec<D>::T;
  griddep_wait();
  const long long u = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (u >= units) return;
  float M = -INFINITY;
  for (int p0 = 0; p0 < P; p0 += 32) {
    const int p = p0 + lane;
    if (p < P) M = fmaxf(M, __ldg(pl + (long long)p * units + u) * kLog2e);
  }
  M = warp_max(M);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M > -INFINITY) {
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      const float lp = p < P ? __ldg(pl + (long long)p * units + u) * kLog2e : -INFINITY;
      unsigned live = __ballot_sync(0xffffffffu, lp > -INFINITY);
      while (live) {  // non-empty partials of this group, four loads in flight at a time
        float w[4];
        V x[4];
        int n = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[q] = 0.f;
          if (live) {
            const int j = __ffs(live) - 1;
            live &= live - 1;
            w[q] = exp2f(__shfl_sync(0xffffffffu, lp, j) - M);
            x[q] = __ldg(reinterpret_cast<const V*>(po + ((long long)(p0 + j) * units + u) * D + lane * E));
            n = q + 1;
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q < n) {
            wsum += w[q];
            MergeVec<D>::fma(acc, w[q], x[q]);
          }
      }
    }
  }
  merge_store<D, BF16_OUT>(out, out_lse, u, lane, acc, wsum, M);
}

}  // namespace
}  // namespace cpattn

// ============================================================================ C ABI
// The merge is launched as a programmatic dependent of whatever kernel precedes it on the
// stream (normally the partials' producer): its CTAs may be scheduled while that kernel's last
// CTAs finish and wait in griddep_wait() for its completion.
template <typename... K, typename... A>
static cudaError_t launch_after_producer(void (*kern)(K...), unsigned grid, cudaStream_t s,
                                         A... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

extern "C" {

const char* cp_status_string(int32_t st) {
  switch (st) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED";
    case CP_ERR_CUDA: return "CP_ERR_CUDA";
    case CP_ERR_TIMEOUT: return "CP_ERR_TIMEOUT";
    case CP_ERR_DEVICE_BOUNDS: return "CP_ERR_DEVICE_BOUNDS";
    default: return "CP_ERR_UNKNOWN";
  }
}

int32_t cp_last_error(char* buf, size_t n) {
  if (buf && n) {
    strncpy(buf, g_detail, n - 1);
    buf[n - 1] = '\0';
  }
  return g_status;
}

int32_t cp_last_error_detail(char* buf, size_t n) { return cp_last_error(buf, n); }

int32_t cp_abi_version(void) { return CPATTN_ABI_VERSION; }
size_t cp_prefill_args_size(void) { return sizeof(cp_prefill_args); }
size_t cp_decode_args_size(void) { return sizeof(cp_decode_args); }

cp_status cp_partition(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                       int32_t cp, int32_t* perm, int32_t* inv_perm, int32_t* shard_offsets,
                       int32_t* chunk_bounds, void* stream) {
  REQUIRE(num_seqs >= 1, "num_seqs must be >= 1 (got %d)", num_seqs);
  REQUIRE(total_tokens >= 0, "total_tokens must be >= 0");
  REQUIRE(cp >= 1 && cp <= 64, "cp must be in [1, 64] (got %d)", cp);
  REQUIRE((long long)num_seqs * cp <= 16384, "num_seqs * cp must be <= 16384");
  REQUIRE(cu_seqlens != nullptr, "cu_seqlens is null");
  REQUIRE(perm || inv_perm || shard_offsets || chunk_bounds, "no output requested");
  const size_t smem = ((size_t)cp * (num_seqs + 1) + cp + 1) * sizeof(int32_t);
  const int threads = 256;
  int blocks = (total_tokens + threads - 1) / threads;
  blocks = blocks < 1 ? 1 : (blocks > 1184 ? 1184 : blocks);
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(cpattn::partition_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (e != cudaSuccess) return launched(e, "cp_partition attribute");
  cpattn::partition_kernel<<<blocks, threads, smem, as_stream(stream)>>>(
      cu_seqlens, num_seqs, total_tokens, cp, perm, inv_perm, shard_offsets, chunk_bounds);
  return launched(cudaGetLastError(), "cp_partition launch");
}

cp_status cp_kv_interleave_layout(const int32_t* cu_seq_lens, int32_t num_seqs,
                                  int32_t total_tokens, int32_t cp, int32_t interleave,
                                  int32_t block_size, const int32_t* block_tables,
                                  int32_t max_blocks, int32_t* local_lens, int32_t* rank_of_token,
                                  int32_t* local_of_token, int64_t* slot_of_token, int32_t* err,
                                  void* stream) {
  REQUIRE(num_seqs >= 1 && total_tokens >= 0, "bad num_seqs / total_tokens");
  REQUIRE(cp >= 1 && cp <= 64, "cp must be in [1, 64] (got %d)", cp);
  REQUIRE(interleave >= 1, "interleave must be >= 1");
  REQUIRE(block_size >= 1, "block_size must be >= 1");
  REQUIRE(cu_seq_lens != nullptr, "cu_seq_lens is null");
  REQUIRE(!slot_of_token || (block_tables && max_blocks >= 1),
          "slot_of_token needs block_tables and max_blocks >= 1");
  REQUIRE(local_lens || rank_of_token || local_of_token || slot_of_token, "no output requested");
  const long long items = total_tokens > (long long)cp * num_seqs ? total_tokens : (long long)cp * num_seqs;
  int blocks = (int)((items + 255) / 256);
  blocks = blocks < 1 ? 1 : (blocks > 4096 ? 4096 : blocks);
  cpattn::interleave_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
      cu_seq_lens, num_seqs, total_tokens, cp, interleave, block_size, block_tables, max_blocks,
      local_lens, rank_of_token, local_of_token, slot_of_token, err);
  return launched(cudaGetLastError(), "cp_kv_interleave_layout launch");
}

int32_t cp_select_prefill_mode(int64_t q_len, int64_t kv_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t elem_bytes) {
  (void)head_dim;
  (void)elem_bytes;
  // Measured on one GB300: the partials + merge step of each mode (pass-KV over contiguous
  // cached + new kv, pass-Q over the paged round-robin cache; cp = 4, d = 128, bf16, batch
  // 8192 / q_len sequences, median of 8 runs with L2 flushed) over q_len in {256, 1024, 4096},
  // kv_len / q_len in {1, 2, 4, .., 32} and G in {1, 2, 4, 8}.  Bit r of kPassQ[G][q] marks
  // the kv_len / q_len = 2^r shapes where pass-Q was faster by more than 3%; everywhere else
  // pass-KV was faster or within 3%.  A shape is looked up at its nearest grid point (log2).
  static const unsigned char kPassQ[4][3] = {
      {0x02, 0x00, 0x0F},  // G = 1: q_len 256, 1024, 4096
      {0x02, 0x00, 0x00},  // G = 2
      {0x02, 0x00, 0x00},  // G = 4
      {0x02, 0x00, 0x00},  // G = 8 (and above)
  };
  if (q_len <= 0 || kv_len < q_len || num_kv_heads <= 0 || num_q_heads < num_kv_heads)
    return CP_PASS_KV;
  auto bucket = [](double x, double per_step, int top) {
    const long i = lround(log2(x) / per_step);
    return (int)(i < 0 ? 0 : (i > top ? top : i));
  };
  const int gi = bucket((double)(num_q_heads / num_kv_heads), 1.0, 3);
  const int qi = bucket((double)q_len / 256.0, 2.0, 2);
  const int ri = bucket((double)kv_len / (double)q_len, 1.0, 5);
  return ((kPassQ[gi][qi] >> ri) & 1) ? CP_PASS_Q : CP_PASS_KV;
}

cp_status cp_kv_cache_write(const void* k_new, const void* v_new, const int32_t* cu_new,
                           const int32_t* start_pos, int32_t num_seqs, int32_t total_new,
                           int32_t num_kv_heads, int32_t head_dim, int32_t dtype, int32_t cp,
                           int32_t interleave, int32_t block_size, const int32_t* block_tables,
                           int32_t max_blocks, int64_t pool_pages, void* k_cache, void* v_cache,
                           int32_t* err, void* stream) {
  REQUIRE(num_seqs >= 1 && total_new >= 0 && num_kv_heads >= 1, "bad sizes");
  REQUIRE(dtype == CP_F32 || dtype == CP_BF16, "dtype must be CP_F32 or CP_BF16");
  REQUIRE(head_dim >= 8 && head_dim % 8 == 0, "head_dim must be a positive multiple of 8");
  REQUIRE(cp >= 1 && cp <= 64 && interleave >= 1 && block_size >= 1, "bad cp / interleave / block_size");
  REQUIRE(max_blocks >= 1 && pool_pages >= 1, "max_blocks and pool_pages must be >= 1");
  REQUIRE(cu_new && start_pos && block_tables, "cu_new, start_pos and block_tables are required");
  REQUIRE_PTR(k_new);
  REQUIRE_PTR(v_new);
  REQUIRE_PTR(k_cache);
  REQUIRE_PTR(v_cache);
  if (total_new == 0) return ok();
  const int esz = dtype == CP_BF16 ? 2 : 4;
  const int vecs = head_dim * esz / 16;
  const long long items = (long long)total_new * num_kv_heads * vecs;
  int blocks = (int)((items + 255) / 256);
  blocks = blocks > 8 * 1184 ? 8 * 1184 : blocks;
  cpattn::kv_write_kernel<<<blocks, 256, 0, as_stream(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), cu_new, start_pos, num_seqs,
      total_new, num_kv_heads, vecs, cp, interleave, block_size, block_tables, max_blocks,
      pool_pages, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), err);
  return launched(cudaGetLastError(), "cp_kv_cache_write launch");
}

cp_status cp_lse_merge(const float* partial_out, const float* partial_lse, int32_t num_partials,
                       int64_t rows, int32_t num_heads, int32_t head_dim, void* out,
                       int32_t out_dtype, float* out_lse, void* stream) {
  REQUIRE(num_partials >= 1, "num_partials must be >= 1");
  REQUIRE(rows >= 0 && num_heads >= 1, "bad rows / num_heads");
  REQUIRE(head_dim == 64 || head_dim == 128, "head_dim must be 64 or 128 (got %d)", head_dim);
  REQUIRE(out_dtype == CP_F32 || out_dtype == CP_BF16, "out_dtype must be CP_F32 or CP_BF16");
  REQUIRE_PTR(partial_out);
  REQUIRE(partial_lse != nullptr, "partial_lse is null");
  REQUIRE_PTR(out);
  const long long units = rows * (long long)num_heads;
  if (units == 0) return ok();
  const long long blocks = (units * 32 + 255) / 256;
  REQUIRE(blocks < (1ll << 31), "too many rows");
  cudaStream_t s = as_stream(stream);
  const unsigned nb = (unsigned)blocks;
  const unsigned nbs = (unsigned)((units + 8ll * cpattn::kMergeUnits - 1) / (8ll * cpattn::kMergeUnits));
#define CP_MERGE_SMALL(D, BF)                                                                 \
  switch (num_partials) {                                                                   \
    case 1: e = launch_after_producer(cpattn::merge_small_kernel<D, BF, 1>, nbs, s, partial_out, partial_lse, units, out, out_lse); break; \
    case 2: e = launch_after_producer(cpattn::merge_small_kernel<D, BF, 2>, nbs, s, partial_out, partial_lse, units, out, out_lse); break; \
    case 3: e = launch_after_producer(cpattn::merge_small_kernel<D, BF, 3>, nbs, s, partial_out, partial_lse, units, out, out_lse); break; \
    case 4: e = launch_after_producer(cpattn::merge_small_kernel<D, BF, 4>, nbs, s, partial_out, partial_lse, units, out, out_lse); break; \
    case 8: e = launch_after_producer(cpattn::merge_small_kernel<D, BF, 8>, nbs, s, partial_out, partial_lse, units, out, out_lse); break; \
    default: e = launch_after_producer(cpattn::merge_kernel<D, BF>, nb, s, partial_out, partial_lse, (int)num_partials, units, out, out_lse); \
  }
  cudaError_t e = cudaSuccess;
  if (head_dim == 128) {
    if (out_dtype == CP_BF16) { CP_MERGE_SMALL(128, true) } else { CP_MERGE_SMALL(128, false) }
  } else {
    if (out_dtype == CP_BF16) { CP_MERGE_SMALL(64, true) } else { CP_MERGE_SMALL(64, false) }
  }
#undef CP_MERGE_SMALL
  if (e == cudaSuccess) e = cudaGetLastError();
  return launched(e, "cp_lse_merge launch");
}

// The kv operands of a prefill call: contiguous k / v (PASS_KV, optionally with their own
// per-sequence lengths) or the paged round-robin pools (PASS_Q).
static cp_status check_kv_source(const cp_prefill_args* a) {
  if (a->mode == CP_PASS_KV) {
    REQUIRE_PTR(a->k);
    REQUIRE_PTR(a->v);
    if (a->cu_seqlens_kv != nullptr) {
      REQUIRE(a->total_kv >= 0, "total_kv must be >= 0");
      REQUIRE(a->total_kv > 0 || a->total_q == 0,
              "total_kv = 0 with %d query rows: every sequence with queries needs at least as "
              "many kv tokens", a->total_q);
    }
  } else {
    REQUIRE_PTR(a->k_cache);
    REQUIRE_PTR(a->v_cache);
    REQUIRE(a->cu_seqlens_kv == nullptr, "cu_seqlens_kv is a PASS_KV argument (PASS_Q takes seq_lens_kv)");
    REQUIRE(a->block_tables != nullptr && a->seq_lens_kv != nullptr,
            "PASS_Q needs block_tables and seq_lens_kv");
    REQUIRE(a->max_blocks >= 1 && a->pool_pages >= 1, "PASS_Q needs max_blocks, pool_pages >= 1");
    REQUIRE(a->interleave >= 1, "interleave must be >= 1");
    if (a->block_size != 16)
      return fail(CP_ERR_UNSUPPORTED, "block_size must be 16 (got %d)", a->block_size);
  }
  return CP_OK;
}

cp_status cp_partial_attn_prefill(const cp_prefill_args* a, void* stream) {
  REQUIRE(a != nullptr, "args is null");
  REQUIRE(a->mode == CP_PASS_KV || a->mode == CP_PASS_Q, "mode must be CP_PASS_KV or CP_PASS_Q");
  REQUIRE(a->dtype == CP_F32 || a->dtype == CP_BF16, "dtype must be CP_F32 or CP_BF16");
  REQUIRE(a->impl >= CP_IMPL_AUTO && a->impl <= CP_IMPL_TCGEN05_SINGLE, "unknown impl %d", a->impl);
  REQUIRE(a->num_seqs >= 1, "num_seqs must be >= 1");
  REQUIRE(a->num_kv_heads >= 1 && a->num_q_heads >= a->num_kv_heads &&
              a->num_q_heads % a->num_kv_heads == 0,
          "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", a->num_q_heads,
          a->num_kv_heads);
  if (a->head_dim != 64 && a->head_dim != 128)
    return fail(CP_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", a->head_dim);
  REQUIRE(a->cp >= 1 && a->cp <= 64, "cp must be in [1, 64] (got %d)", a->cp);
  REQUIRE(a->total_q >= 0 && a->max_seqlen_q >= 0, "total_q / max_seqlen_q must be >= 0");
  REQUIRE(a->q_shard >= -1 && a->q_shard < a->cp, "q_shard out of range");
  REQUIRE(a->kv_shard >= -1 && a->kv_shard < a->cp, "kv_shard out of range");
  REQUIRE(a->debug == 0 || a->debug == 1, "debug must be 0 or 1");
  REQUIRE(a->cu_seqlens_q != nullptr, "cu_seqlens_q is null");
  REQUIRE_PTR(a->q);
  REQUIRE_PTR(a->out);
  REQUIRE(a->lse != nullptr, "lse is null");
  const cp_status st = check_kv_source(a);
  if (st != CP_OK) return st;
  if (a->total_q == 0) return ok();
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  int impl = a->impl;
  if (impl == CP_IMPL_AUTO) impl = (a->dtype == CP_BF16 && cp_prefill_tc_supported(*a)) ? CP_IMPL_TCGEN05 : CP_IMPL_SIMT;
  if (impl == CP_IMPL_TCGEN05 || impl == CP_IMPL_TCGEN05_SINGLE) {
    if (a->dtype != CP_BF16 || !cp_prefill_tc_supported(*a))
      return fail(CP_ERR_UNSUPPORTED, "the tcgen05 kernel needs bf16 inputs and a supported shape");
    return launched(cp_launch_prefill_tc(*a, scale, as_stream(stream)), "prefill (tcgen05) launch");
  }
  return launched(cp_launch_prefill_simt(*a, scale, as_stream(stream)), "prefill (simt) launch");
}

// Shape arguments of the fused prefill (those its split plan reads too).
static cp_status check_fused_shape(const cp_prefill_args* a) {
  REQUIRE(a != nullptr, "args is null");
  REQUIRE(a->mode == CP_PASS_KV || a->mode == CP_PASS_Q, "mode must be CP_PASS_KV or CP_PASS_Q");
  if (a->dtype != CP_BF16) return fail(CP_ERR_UNSUPPORTED, "the fused prefill takes bf16 inputs");
  if (a->mode == CP_PASS_Q && a->impl == CP_IMPL_TCGEN05_SINGLE)
    return fail(CP_ERR_UNSUPPORTED, "the fused pass-Q prefill runs on the two-tile kernel only");
  if (a->head_dim != 64 && a->head_dim != 128)
    return fail(CP_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", a->head_dim);
  REQUIRE(a->num_seqs >= 1 && a->num_kv_heads >= 1 && a->num_q_heads >= 1 &&
              a->num_q_heads % a->num_kv_heads == 0,
          "bad head counts");
  REQUIRE(a->cp >= 1 && a->cp <= 64, "cp must be in [1, 64]");
  REQUIRE(a->q_shard == -1 && a->kv_shard == -1, "the fused prefill covers every pair");
  REQUIRE(a->total_q >= 0 && a->max_seqlen_q >= 0, "bad total_q / max_seqlen_q");
  return CP_OK;
}

cp_status cp_prefill_fused_workspace_size(const cp_prefill_args* a, size_t* bytes) {
  REQUIRE(bytes != nullptr, "bytes is null");
  *bytes = 0;
  const cp_status st = check_fused_shape(a);
  if (st != CP_OK) return st;
  *bytes = cp_prefill_fused_split_bytes(*a);
  return ok();
}

cp_status cp_attn_prefill_fused(const cp_prefill_args* a, void* workspace, size_t workspace_bytes,
                                void* out, float* out_lse, void* stream) {
  cp_status st = check_fused_shape(a);
  if (st != CP_OK) return st;
  REQUIRE(a->cu_seqlens_q != nullptr, "cu_seqlens_q is null");
  REQUIRE_PTR(a->q);
  st = check_kv_source(a);
  if (st != CP_OK) return st;
  REQUIRE_PTR(out);
  REQUIRE(out_lse != nullptr, "out_lse is null");
  REQUIRE(a->debug == 0, "debug must be 0");
  REQUIRE(workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
          "workspace must be 256-byte aligned");
  if (a->total_q == 0) return ok();
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  return launched(cp_launch_prefill_fused(*a, scale, out, out_lse, workspace,
                                          workspace ? workspace_bytes : 0, as_stream(stream)),
                  "fused prefill launch");
}

cp_status cp_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t cp, int32_t interleave,
                         int32_t block_size, int32_t max_seq_len, int32_t* num_splits,
                         int32_t* split_tokens) {
  REQUIRE(num_seqs >= 1 && num_kv_heads >= 1 && cp >= 1 && interleave >= 1 && block_size >= 1 &&
              max_seq_len >= 1,
          "all sizes must be >= 1");
  REQUIRE(num_splits && split_tokens, "outputs are null");
  // largest rank share: rank 0 never holds fewer tokens than another rank
  const long long group = (long long)interleave * cp;
  long long rem = max_seq_len % group;
  const long long share = (max_seq_len / group) * interleave + (rem < interleave ? rem : interleave);
  // target ~4096 local tokens per CTA (measured best between 512 and 6144 on the 64-sequence
  // decode workload: fewer CTAs means fewer prologues, partials and, when fused, end-of-CTA
  // fences) and at least ~8 CTAs per SM over 152 SMs in total
  const long long base = (long long)num_seqs * num_kv_heads * cp;
  long long S = (share + 4095) / 4096;
  const long long want = (8ll * 152 + base - 1) / base;
  if (S < want) S = want;
  const long long max_S = (share + block_size - 1) / block_size;
  if (S > max_S) S = max_S;
  if (S < 1) S = 1;
  long long st = (share + S - 1) / S;
  st = (st + block_size - 1) / block_size * block_size;
  S = (share + st - 1) / st;
  REQUIRE(S <= 65535, "too many splits");
  *num_splits = (int32_t)S;
  *split_tokens = (int32_t)st;
  return ok();
}

static cp_status check_decode_args(const cp_decode_args* a, bool need_partials);

cp_status cp_partial_attn_decode(const cp_decode_args* a, void* stream) {
  const cp_status st = check_decode_args(a, true);
  if (st != CP_OK) return st;
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  return launched(cp_launch_decode(*a, scale, as_stream(stream)), "decode launch");
}

cp_status cp_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t cp, int32_t num_splits,
                                   size_t* bytes) {
  REQUIRE(bytes != nullptr, "bytes is null");
  REQUIRE(num_seqs >= 1 && num_q_heads >= 1 && num_kv_heads >= 1 && head_dim >= 1 && cp >= 1 &&
              num_splits >= 1,
          "all sizes must be >= 1");
  size_t ol, oo;
  *bytes = cp_decode_ws_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, cp * num_splits, &ol, &oo);
  return ok();
}

cp_status cp_decode_attention(const cp_decode_args* a, void* workspace, size_t workspace_bytes,
                              void* out, float* out_lse, void* stream) {
  const cp_status st = check_decode_args(a, false);
  if (st != CP_OK) return st;
  REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
          "workspace must be a non-null 256-byte aligned pointer");
  REQUIRE_PTR(out);
  if ((long long)a->cp * a->num_splits > 256)
    return fail(CP_ERR_UNSUPPORTED, "cp * num_splits must be <= 256 for the fused decode (got %d)",
                a->cp * a->num_splits);
  size_t ol, oo;
  const size_t need = cp_decode_ws_layout(a->num_seqs, a->num_q_heads, a->num_kv_heads, a->head_dim,
                                          a->cp * a->num_splits, &ol, &oo);
  REQUIRE(workspace_bytes >= need, "workspace too small: %zu bytes given, %zu needed",
          workspace_bytes, need);
  CpDecodeWorkspace ws;
  ws.counters = static_cast<int32_t*>(workspace);
  ws.partial_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + ol);
  ws.partial_out = reinterpret_cast<float*>(static_cast<char*>(workspace) + oo);
  const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.f / sqrtf((float)a->head_dim);
  return launched(cp_launch_decode_fused(*a, scale, ws, out, out_lse, as_stream(stream)),
                  "fused decode launch");
}

static cp_status check_decode_args(const cp_decode_args* a, bool need_partials) {
  REQUIRE(a != nullptr, "args is null");
  REQUIRE(a->dtype == CP_F32 || a->dtype == CP_BF16, "dtype must be CP_F32 or CP_BF16");
  REQUIRE(a->num_seqs >= 1, "num_seqs must be >= 1");
  REQUIRE(a->num_kv_heads >= 1 && a->num_q_heads % a->num_kv_heads == 0,
          "num_q_heads must be a multiple of num_kv_heads");
  const int G = a->num_q_heads / a->num_kv_heads;
  if (G < 1 || G > (a->dtype == CP_BF16 ? 16 : 8))
    return fail(CP_ERR_UNSUPPORTED, "q heads per kv head must be 1 .. %d for this dtype (got %d)",
                a->dtype == CP_BF16 ? 16 : 8, G);
  if (a->head_dim != 64 && a->head_dim != 128)
    return fail(CP_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", a->head_dim);
  if (a->block_size != 16)
    return fail(CP_ERR_UNSUPPORTED, "block_size must be 16 (got %d)", a->block_size);
  REQUIRE(a->cp >= 1 && a->cp <= 64 && a->interleave >= 1, "bad cp / interleave");
  REQUIRE(a->num_splits >= 1 && a->num_splits <= 65535, "num_splits must be in [1, 65535]");
  REQUIRE(a->split_tokens >= a->block_size && a->split_tokens % a->block_size == 0,
          "split_tokens must be a positive multiple of block_size");
  REQUIRE(a->max_blocks >= 1 && a->pool_pages >= 1, "max_blocks and pool_pages must be >= 1");
  REQUIRE((long long)a->cp * a->num_seqs <= 65535 && a->num_kv_heads <= 65535, "grid too large");
  REQUIRE_PTR(a->q);
  REQUIRE_PTR(a->k_cache);
  REQUIRE_PTR(a->v_cache);
  REQUIRE(a->block_tables && a->seq_lens, "block_tables and seq_lens are required");
  if (need_partials) {
    REQUIRE_PTR(a->out);
    REQUIRE(a->lse != nullptr, "lse is required");
  }
  return ok();
}

}  // extern "C"

// ------------------------------------------------------------------ helpers for other units
cp_status cp_check_decode_args_for_fused(const cp_decode_args* a, const void* out) {
  const cp_status st = check_decode_args(a, false);
  if (st != CP_OK) return st;
  REQUIRE_PTR(out);
  if ((long long)a->cp * a->num_splits > 256)
    return fail(CP_ERR_UNSUPPORTED, "cp * num_splits must be <= 256 for the fused decode (got %d)",
                a->cp * a->num_splits);
  return CP_OK;
}

cp_status cp_fail_detail(cp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  g_status = st;
  return st;
}

cp_status cp_launch_status(cudaError_t e, const char* what) { return launched(e, what); }
