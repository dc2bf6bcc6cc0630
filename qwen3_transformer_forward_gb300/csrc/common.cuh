// Shared device helpers of libqw (GB300, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qw.h"

namespace qw {

using bf16 = __nv_bfloat16;

// Every workspace starts with this many bytes of completion counters; they
// must be zero before the first call and each call leaves them zero.
constexpr size_t kCounterBytes = 64 * 1024;

// Bit of the decode-attention error word set when a context_lens entry exceeds
// the max_context a call was planned for: keys past it are not read, so the
// output misses them.  qw_device_error reports it as QW_ERR_INVALID_ARG.
constexpr unsigned int kErrContextOverflow = 0x100u;

// ---------------------------------------------------------------------------
// element conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// round a float to the storage type and back (the model-dtype rounding)
template <typename T> __device__ __forceinline__ float round_t(float x) { return to_f(from_f<T>(x)); }

// number of elements in one 16-byte vector
template <typename T> struct V16 { static constexpr int N = 16 / sizeof(T); };

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t*>(&h);
}

// Softmax weights p[0..3] of one m16n8k16 A-fragment row (keys 2t, 2t+1,
// 2t+8, 2t+9) as a bf16 pair hi = bf16(p), lo = bf16(p - hi): hi + lo
// represents p to about 2^-17 relative (p - hi is exact in fp32).  a0/a2
// carry hi, a1/a3 carry lo: the fragment's rows r and r + 8.
__device__ __forceinline__ void split_p(const float (&p)[4], uint32_t& a0, uint32_t& a1, uint32_t& a2,
                                        uint32_t& a3) {
  a0 = pack_bf16(p[0], p[1]);
  a2 = pack_bf16(p[2], p[3]);
  a1 = pack_bf16(p[0] - bf16_lo(a0), p[1] - bf16_hi(a0));
  a3 = pack_bf16(p[2] - bf16_lo(a2), p[3] - bf16_hi(a2));
}

// QK-RMSNorm + RoPE of one 128-wide head ([SK] §3, §8 ①), pairing element i
// with i + 64.  Used by the standalone kernel (eight lanes per head) and by the
// QKV GEMM epilogue (one thread per head); every step is an explicit
// round-to-nearest fp32 operation, so no contraction into FMA can make the
// two differ.  Sum of squares: eight partials, partial p over the pairs
// (8p + e, 64 + 8p + e) for e = 0..7 in order, combined as a balanced tree.
__device__ __forceinline__ float qk_ss8(const float (&x1)[8], const float (&x2)[8]) {
  float ss = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = __fadd_rn(ss, __fadd_rn(__fmul_rn(x1[e], x1[e]), __fmul_rn(x2[e], x2[e])));
  return ss;
}
__device__ __forceinline__ float qk_ss_tree(const float (&p)[8]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])),
                   __fadd_rn(__fadd_rn(p[4], p[5]), __fadd_rn(p[6], p[7])));
}
__device__ __forceinline__ float qk_inv_rms(float ss, float eps) {
  return rsqrtf(__fadd_rn(__fmul_rn(ss, 1.0f / 128.0f), eps));
}
// normed (rounded to bf16 as the q_norm / k_norm output) then rotated; zero when the position is invalid
__device__ __forceinline__ void qk_rope_pair(float x1, float x2, float inv, float g1, float g2, float c, float sn,
                                             bool pos_ok, float& y1, float& y2) {
  const float n1 = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(x1, inv), g1)));
  const float n2 = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(x2, inv), g2)));
  y1 = pos_ok ? __fsub_rn(__fmul_rn(n1, c), __fmul_rn(n2, sn)) : 0.0f;
  y2 = pos_ok ? __fadd_rn(__fmul_rn(n2, c), __fmul_rn(n1, sn)) : 0.0f;
}

// 16-byte vector load into floats
__device__ __forceinline__ void load16(const bf16* p, float* f) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void load16(const float* p, float* f) {
  float4 u = *reinterpret_cast<const float4*>(p);
  f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}
__device__ __forceinline__ void store16(bf16* p, const float* f) {
  uint4 u;
  u.x = pack_bf16(f[0], f[1]); u.y = pack_bf16(f[2], f[3]);
  u.z = pack_bf16(f[4], f[5]); u.w = pack_bf16(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store16(float* p, const float* f) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

// ---------------------------------------------------------------------------
// warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async 16 bytes global -> shared (L2 only), with a zero-fill variant
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t saddr, const void* g, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(g), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// thread-block cluster helpers (distributed shared memory)
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory offset in cluster CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ long long ld_cluster_s64(uint32_t addr) {
  long long v;
  asm volatile("ld.shared::cluster.s64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace qw

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel waits for the previous one to finish
// and publish its memory (pdl_wait) before touching anything it produced, and
// then lets the next kernel on the stream start early (pdl_trigger).  Waiting
// first keeps at most one kernel parked ahead: measured on the 28-layer
// decode step, triggering before the wait let chains of waiting CTAs occupy
// the SMs and cost about 5%.  Both are no-ops without the launch attribute.
// ---------------------------------------------------------------------------
namespace qw {
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
}  // namespace qw

// ---------------------------------------------------------------------------
// host-side error reporting shared by every entry point (defined in qw_api.cu)
// ---------------------------------------------------------------------------
namespace qw {
// Paged KV cache: key position p of sequence s sits at row
// table[s * max_blocks + p / block_size] * block_size + p % block_size.
// table == nullptr: rows are contiguous from the sequence's base row.
struct KvPages {
  const int32_t* table;
  int max_blocks;
  int block_size;
};

int set_error(int code, const char* fmt, ...);
int check_launch(const char* what);
bool pdl_enabled();   // programmatic dependent launch on (default) unless QW_NO_PDL=1

// Launches `kern` on `st` with programmatic stream serialization (when enabled).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
}  // namespace qw
