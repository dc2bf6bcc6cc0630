// Temperature / top-p sampling of one token per logits row (the Sampler that
// nano-vllm compiles with the other small operators, [SK] §3).  The pages give
// no semantics; the reading implemented here:
//   T == 0 (or negative, or NaN): greedy, argmax with the lowest index on ties;
//   otherwise the token is drawn from softmax(logits / T) restricted to the
//   nucleus: the row's distinct logit values are taken from the largest down
//   until their softmax mass reaches P of the row's mass, and every token whose
//   logit is at least that last value is kept (ties at the boundary all kept);
//   the draw is argmax over the nucleus of logits / T + G, G = -log(-log u),
//   the Gumbel-max identity, with the caller's uniforms u in (0, 1).
//
// bf16 logits take at most 65536 distinct values, so the nucleus boundary is
// found exactly from a histogram of the logits' 16-bit order-preserving keys:
//   sample_hist_kernel   grid (chunks, B): a shared-memory histogram of one
//                        chunk (two 16-bit counts per 32-bit word), merged into
//                        the row's global histogram with atomics; the row max
//   sample_nucleus_kernel  one CTA per row: mass of each key = count x
//                        exp((value - max) / T), scanned from the largest key
//                        down to the first key where the running mass reaches
//                        P of the total; the histogram is zeroed again
//   sample_draw_kernel   grid (chunks, B): the Gumbel-max argmax of each chunk
//                        over the nucleus; the row's last CTA (completion
//                        counter) merges the chunk winners in chunk order
// Every reduction runs in a fixed order, so results do not depend on timing.
// Traffic per row: the logits twice and the uniforms once (HBM or L2), the
// 256 KB histogram once read and once cleared.
#include <math.h>

#include "common.cuh"

namespace qw {
namespace smp {

constexpr int CHUNK = 8192;          // logits per CTA of the chunked kernels
constexpr int THREADS = 256;
constexpr int NKEYS = 65536;         // distinct bf16 bit patterns
constexpr int NUC_THREADS = 1024;
constexpr int KEYS_PER_THREAD = NKEYS / NUC_THREADS;
constexpr size_t HIST_SMEM = size_t(NKEYS / 2) * sizeof(uint32_t);   // 128 KB

// order-preserving key of a bf16 bit pattern (larger value -> larger key); -0 maps to +0
__device__ __forceinline__ uint32_t key_of(uint32_t bits) {
  bits &= 0xFFFFu;
  if (bits == 0x8000u) bits = 0u;
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}
__device__ __forceinline__ float value_of(uint32_t key) {
  const uint32_t bits = (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
  return __uint_as_float(bits << 16);
}
__device__ __forceinline__ bool greedy_temp(float T) { return !(T > 0.0f); }   // T <= 0 or NaN

struct Ws {
  unsigned int* counters;   // [B] completion counters (first 64 KiB of the workspace)
  uint32_t* hist;           // [B][65536]
  uint32_t* row_max;        // [B] largest key of the row (0 = not yet seen)
  uint32_t* boundary;       // [B] smallest key in the nucleus
  float2* partial;          // [B][chunks] (score, index as float bits)
};

__global__ void __launch_bounds__(THREADS, 1) sample_hist_kernel(const bf16* __restrict__ logits, int64_t V,
                                                                  int chunks, const float* __restrict__ temperature,
                                                                  Ws ws) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint32_t sh[];   // [32768] two 16-bit counts per word
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
  if (greedy_temp(temperature[b])) return;   // uniform over the CTA
  for (int i = tid; i < NKEYS / 2; i += THREADS) sh[i] = 0u;
  __syncthreads();
  const int64_t lo = int64_t(c) * CHUNK, hi = min(V, lo + CHUNK);
  const bf16* row = logits + int64_t(b) * V;
  uint32_t kmax = 0u;
  for (int64_t i = lo + int64_t(tid) * 8; i < hi; i += int64_t(THREADS) * 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + i);   // V % 8 == 0: whole vectors only
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t k = key_of(e & 1 ? w[e >> 1] >> 16 : w[e >> 1]);
      kmax = max(kmax, k);
      atomicAdd(&sh[k >> 1], (k & 1u) ? 0x10000u : 1u);   // a chunk holds < 65536 of any key
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  if ((tid & 31) == 0) atomicMax(&ws.row_max[b], kmax);
  __syncthreads();
  uint32_t* gh = ws.hist + int64_t(b) * NKEYS;
  for (int i = tid; i < NKEYS / 2; i += THREADS) {
    const uint32_t w = sh[i];
    if (w & 0xFFFFu) atomicAdd(&gh[2 * i], w & 0xFFFFu);
    if (w >> 16) atomicAdd(&gh[2 * i + 1], w >> 16);
  }
}

__global__ void __launch_bounds__(NUC_THREADS) sample_nucleus_kernel(const float* __restrict__ temperature,
                                                                      const float* __restrict__ top_p, Ws ws) {
  pdl_wait();
  pdl_trigger();
  __shared__ float warp_sum[NUC_THREADS / 32];
  __shared__ uint32_t found;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float T = temperature[b];
  if (greedy_temp(T)) return;
  float P = top_p[b];
  P = P > 0.0f ? fminf(P, 1.0f) : 1.0f;   // P outside (0, 1] (or NaN): the whole row
  const float vmax = value_of(ws.row_max[b]);
  uint32_t* gh = ws.hist + int64_t(b) * NKEYS;
  auto mass = [&](int j, uint32_t cnt) {   // softmax mass (unnormalised) of key k0 - j
    return float(cnt) * expf((value_of(uint32_t(NKEYS - 1 - tid * KEYS_PER_THREAD - j)) - vmax) / T);
  };
  // thread t owns keys 65535 - 64t down to 65535 - 64t - 63 (descending values)
  const int k0 = NKEYS - 1 - tid * KEYS_PER_THREAD;
  float local = 0.0f;
  for (int j = 0; j < KEYS_PER_THREAD; ++j) {
    const uint32_t c = gh[k0 - j];
    if (c) local += mass(j, c);
  }
  // scan of the per-thread masses in thread order (= descending values).  This
  // thread's interval is (E, I]; E is the previous lane's inclusive value and
  // the warp prefixes are running sums, so the intervals tile [0, total] exactly.
  float inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  float inc_prev = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) inc_prev = 0.0f;
  if (lane == 31) warp_sum[warp] = inc;
  if (tid == 0) found = 0xFFFFFFFFu;
  __syncthreads();
  float wprefix = 0.0f, total = 0.0f;
  for (int w = 0; w < NUC_THREADS / 32; ++w) {
    if (w == warp) wprefix = total;
    total += warp_sum[w];
  }
  const float E = wprefix + inc_prev, I = wprefix + inc;
  const float target = P * total;
  if (E < target && target <= I) atomicMin(&found, uint32_t(tid));
  __syncthreads();
  if (uint32_t(tid) == found) {   // walk this thread's keys to the one where the running mass reaches the target
    float c = 0.0f;
    int hit = -1, last_nz = 0;
    for (int j = 0; j < KEYS_PER_THREAD; ++j) {
      const uint32_t n = gh[k0 - j];
      if (!n) continue;
      c += mass(j, n);
      last_nz = j;
      if (E + c >= target) {
        hit = j;
        break;
      }
    }
    // (the walk's running sum can fall an ulp short of the scan's: the range's last key then)
    ws.boundary[b] = uint32_t(k0 - (hit >= 0 ? hit : last_nz));
  }
  // leave the histogram and the row max zero for the next call
  for (int j = 0; j < KEYS_PER_THREAD; ++j)
    if (gh[k0 - j]) gh[k0 - j] = 0u;
  __syncthreads();
  if (tid == 0) ws.row_max[b] = 0u;
}

// better (score, index): larger score, then lower index
__device__ __forceinline__ void take_best(float& s, int& i, float s2, int i2) {
  if (s2 > s || (s2 == s && i2 < i)) {
    s = s2;
    i = i2;
  }
}

__global__ void __launch_bounds__(THREADS) sample_draw_kernel(const bf16* __restrict__ logits, int64_t V, int chunks,
                                                              const float* __restrict__ temperature,
                                                              const float* __restrict__ uniforms,
                                                              int64_t* __restrict__ out, Ws ws) {
  pdl_wait();
  pdl_trigger();
  __shared__ float ws_s[THREADS / 32];
  __shared__ int ws_i[THREADS / 32];
  __shared__ int is_last;
  const int b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float T = temperature[b];
  const bool greedy = greedy_temp(T);
  const uint32_t kb = greedy ? 0u : ws.boundary[b];
  const int64_t lo = int64_t(c) * CHUNK, hi = min(V, lo + CHUNK);
  const bf16* row = logits + int64_t(b) * V;
  const float* urow = uniforms + int64_t(b) * V;
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int64_t i = lo + int64_t(tid) * 8; i < hi; i += int64_t(THREADS) * 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float4 ua = make_float4(0.f, 0.f, 0.f, 0.f), ub = ua;
    if (!greedy) {
      ua = *reinterpret_cast<const float4*>(urow + i);
      ub = *reinterpret_cast<const float4*>(urow + i + 4);
    }
    const float uu[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t bits = (e & 1 ? w[e >> 1] >> 16 : w[e >> 1]) & 0xFFFFu;
      const float l = __uint_as_float(bits << 16);
      float s;
      if (greedy) {
        s = l;
      } else {
        if (key_of(bits) < kb) continue;
        const float uc = fminf(fmaxf(uu[e], 5.9604645e-8f), 0.99999994f);   // [2^-24, 1 - 2^-24]
        s = l / T - logf(-logf(uc));
      }
      take_best(best, bi, s, int(i) + e);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    take_best(best, bi, s2, i2);
  }
  if (lane == 0) {
    ws_s[warp] = best;
    ws_i[warp] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < THREADS / 32; ++w) take_best(best, bi, ws_s[w], ws_i[w]);
    ws.partial[int64_t(b) * chunks + c] = make_float2(best, __int_as_float(bi));
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ws.counters + b) : "memory");
    is_last = old == unsigned(chunks - 1);
  }
  __syncthreads();
  if (is_last && tid == 0) {   // the row's chunk winners in chunk order
    float s = -INFINITY;
    int idx = 0x7FFFFFFF;
    for (int k = 0; k < chunks; ++k) {
      const float2 p = __ldcg(ws.partial + int64_t(b) * chunks + k);
      take_best(s, idx, p.x, __float_as_int(p.y));
    }
    out[b] = idx == 0x7FFFFFFF ? 0 : int64_t(idx);
    ws.counters[b] = 0u;
  }
}

inline int n_chunks(int64_t V) { return int((V + CHUNK - 1) / CHUNK); }

inline size_t workspace_bytes(int64_t B, int64_t V) {
  return kCounterBytes + size_t(B) * NKEYS * 4 + size_t(B) * 8 + size_t(B) * n_chunks(V) * sizeof(float2);
}

}  // namespace smp
}  // namespace qw

using namespace qw;

extern "C" size_t qw_sample_workspace_size(int64_t B, int64_t V) {
  if (B <= 0 || V <= 0) return 0;
  return smp::workspace_bytes(B, V);
}

extern "C" int qw_sample(const void* logits, int64_t B, int64_t V, const float* temperature, const float* top_p,
                         const float* uniforms, int64_t* out, void* workspace, size_t workspace_bytes, int dtype,
                         void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_sample: bf16 logits only");
  if (B < 0 || V <= 0 || V % 8 || V > (int64_t(1) << 30))
    return set_error(QW_ERR_INVALID_ARG, "qw_sample: V must be a positive multiple of 8 below 2^30");
  if (B == 0) return QW_OK;
  if (size_t(B) * sizeof(unsigned int) > kCounterBytes)
    return set_error(QW_ERR_SHAPE, "qw_sample: %lld rows exceed the counter area", (long long)B);
  if (!logits || !temperature || !top_p || !uniforms || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_sample: null pointer");
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(uniforms)) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_sample: logits and uniforms must be 16-byte aligned");
  const size_t need = smp::workspace_bytes(B, V);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 16)
    return set_error(QW_ERR_WORKSPACE, "qw_sample: 16-byte aligned workspace of %zu bytes needed", need);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(smp::sample_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smp::HIST_SMEM));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  uint8_t* base = static_cast<uint8_t*>(workspace);
  smp::Ws ws;
  ws.counters = reinterpret_cast<unsigned int*>(base);
  ws.hist = reinterpret_cast<uint32_t*>(base + kCounterBytes);
  ws.row_max = ws.hist + size_t(B) * smp::NKEYS;
  ws.boundary = ws.row_max + B;
  ws.partial = reinterpret_cast<float2*>(ws.boundary + B);
  const int chunks = smp::n_chunks(V);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bf16* lg = static_cast<const bf16*>(logits);
  launch_pdl(smp::sample_hist_kernel, dim3(unsigned(chunks), unsigned(B)), smp::THREADS, smp::HIST_SMEM, st, lg, V,
             chunks, temperature, ws);
  int rc = check_launch("sample_hist_kernel");
  if (rc) return rc;
  launch_pdl(smp::sample_nucleus_kernel, dim3(unsigned(B)), smp::NUC_THREADS, 0, st, temperature, top_p, ws);
  rc = check_launch("sample_nucleus_kernel");
  if (rc) return rc;
  launch_pdl(smp::sample_draw_kernel, dim3(unsigned(chunks), unsigned(B)), smp::THREADS, 0, st, lg, V, chunks,
             temperature, uniforms, out, ws);
  return check_launch("sample_draw_kernel");
}
