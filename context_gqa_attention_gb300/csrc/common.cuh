// Shared device/host helpers of libcpattn (internal; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/cpattn.h"

#define CP_DEV __device__ __forceinline__

namespace cpattn {

// First device-side error wins; CP_OK is never written.
CP_DEV void report(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static CP_DEV float to_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static CP_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
};

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start while the previous kernel on the stream finishes; it waits here, before reading what
// that kernel wrote, until the previous grid has completed and its writes are visible (no-op
// for a normal launch).  The previous kernel may let it start early (launch_dependents) once
// its CTAs have issued their last loads.
CP_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
CP_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Chunk bounds of the load-balanced partition: b_k = floor(k*T/(2cp)).
CP_DEV int chunk_bound(int k, int T, int cp) {
  // k, T >= 0; 32-bit division whenever k*T fits (64-bit division is a long software routine)
  const unsigned long long num = (unsigned long long)k * (unsigned)T;
  const unsigned den = 2u * (unsigned)cp;
  if (num <= 0xffffffffull) return (int)((unsigned)num / den);
  return (int)(num / den);
}

// Chunk index c (0..2cp-1) of within-sequence offset t (0 <= t < T).
CP_DEV int chunk_of(int t, int T, int cp) {
  const unsigned long long num = (unsigned long long)t * (2u * (unsigned)cp);
  int c = num <= 0xffffffffull ? (int)((unsigned)num / (unsigned)T)  // lower estimate
                               : (int)(num / (unsigned)T);
  // b_c <= t < b_{c+1}; the estimate is within one of the answer.
  while (c + 1 < 2 * cp && chunk_bound(c + 1, T, cp) <= t) ++c;
  while (c > 0 && chunk_bound(c, T, cp) > t) --c;
  return c;
}

CP_DEV int shard_of_chunk(int c, int cp) { return c < cp ? c : 2 * cp - 1 - c; }

// Round-robin interleave: tokens of rank r among positions [0, L).
CP_DEV int rank_local_len(long long L, int r, int cp, int I) {
  if (L >= 0 && L <= 0x7fffffffll && (long long)I * cp <= 0x7fffffffll) {  // 32-bit division
    const unsigned g = (unsigned)I * (unsigned)cp, l = (unsigned)L;
    const int rem = (int)(l % g) - r * I;
    return (int)(l / g) * I + (rem < 0 ? 0 : (rem > I ? I : rem));
  }
  long long group = (long long)I * cp;
  long long full = (L / group) * I;
  long long rem = L % group - (long long)r * I;
  rem = rem < 0 ? 0 : (rem > I ? I : rem);
  return (int)(full + rem);
}

// Sequence of a row: largest b with cu[b] <= row (cu non-decreasing, cu[0] = 0).
CP_DEV int seq_of_row(const int32_t* __restrict__ cu, int num_seqs, int row) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

CP_DEV float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
CP_DEV float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace cpattn

// ---------------------------------------------------------------------------- launchers
// Implemented in the kernel translation units; called by the host ABI in api.cu after
// argument validation.  They return the launch status.
cudaError_t cp_launch_prefill_simt(const cp_prefill_args& a, float scale, cudaStream_t s);
cudaError_t cp_launch_prefill_tc(const cp_prefill_args& a, float scale, cudaStream_t s);
// ws / ws_bytes: scratch for the fused pass-Q tail split (NULL or too small: no split)
cudaError_t cp_launch_prefill_fused(const cp_prefill_args& a, float scale, void* out, float* lse,
                                    void* ws, size_t ws_bytes, cudaStream_t s);
// Scratch bytes the fused prefill's tail split wants on the current device (0: no split).
size_t cp_prefill_fused_split_bytes(const cp_prefill_args& a);
bool cp_prefill_tc_supported(const cp_prefill_args& a);
cudaError_t cp_launch_decode(const cp_decode_args& a, float scale, cudaStream_t s);
// 2D bf16 TMA descriptor (CUtensorMap, 64-byte aligned storage of 128 bytes) over `rows` rows
// of `cols` elements, box of 64 columns x box_rows rows, 128-byte swizzle, zero fill.
bool cp_make_bf16_map_2d(void* map, const void* base, unsigned long long cols,
                         unsigned long long rows, unsigned long long pitch_elems,
                         unsigned box_rows);
// 3D bf16 TMA descriptor over a paged pool of `rows` rows of d = 128 elements seen as
// {64 columns, rows, 2 column halves}: one box {64, 16, 2} is a whole 16-row page, landing in
// shared memory as [half][16 rows][128 bytes] (128-byte swizzle).  False if the driver refuses.
bool cp_make_bf16_page_map(void* map, const void* base, unsigned long long rows);
// 4D variant for MMA operands: {64 columns, 8 rows, 2 halves, rows / 8 row groups}, box
// {64, 8, 2, 2} = one 16-row page landing as [row group][half][8 rows][128 bytes], so that
// consecutive 8-row groups of consecutive pages sit a uniform 2 KB apart.
bool cp_make_bf16_page_map4(void* map, const void* base, unsigned long long rows);

// Scratch of the fused decode: arrival counters [B][Hkv] (zero between calls), partial LSEs
// [cp*S][B][Hq] and partial outputs [cp*S][B][Hq][d], each region 256-byte aligned.
struct CpDecodeWorkspace {
  int32_t* counters;
  float* partial_lse;
  float* partial_out;
};
inline size_t cp_align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline size_t cp_decode_ws_layout(int B, int Hq, int Hkv, int d, int P, size_t* off_lse,
                                  size_t* off_out) {
  const size_t c = cp_align256((size_t)B * Hkv * sizeof(int32_t));
  const size_t l = cp_align256((size_t)P * B * Hq * sizeof(float));
  const size_t o = cp_align256((size_t)P * B * Hq * d * sizeof(float));
  *off_lse = c;
  *off_out = c + l;
  return c + l + o;
}
cudaError_t cp_launch_decode_fused(const cp_decode_args& a, float scale, const CpDecodeWorkspace& ws,
                                   void* out, float* out_lse, cudaStream_t s);

// Host helpers exported by api.cu for entry points defined in other translation units.
cp_status cp_check_decode_args_for_fused(const cp_decode_args* a, const void* out);
cp_status cp_fail_detail(cp_status st, const char* fmt, ...);
cp_status cp_launch_status(cudaError_t e, const char* what);
