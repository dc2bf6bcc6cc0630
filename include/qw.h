/*
 * qw.h - C ABI of the GB300 (sm_103a) Qwen3 forward hot path.
 *
 * One shared library, libqw.so, exposes the steps of a nano-vllm-style
 * Qwen3 forward pass: the vocab-sharded embedding, fused residual add +
 * RMSNorm, the linear layers (merged QKV and gate_up column splits, o_proj
 * and down_proj row splits), per-head QK-RMSNorm + RoPE + KV-cache store,
 * causal GQA attention for prefill and decode, SiluAndMul and the
 * vocab-sharded lm_head with greedy argmax.
 *
 * Sources, cited by page and section:
 *   [VH]  devpress page "vocab 切 / head 切" (nano-vllm tensor parallelism):
 *         §3 VocabParallelEmbedding, §4 ParallelLMHead, §5 head split and
 *         KV cache, §6 sharded == single-card check.
 *   [TP]  devpress page on tensor-parallel maths: §3 column vs row split,
 *         §4 the two column->row pairs, §5 embedding/LM head, §6 RMSNorm.
 *   [VPE] "从零实现 vLLM (1.1): 并行词嵌入 VocabParallelEmbedding".
 *   [SK]  "3.3 模型骨架与核心算子" (AIInfraGuide): §1 decoder layer,
 *         §2 RMSNorm, §3 RoPE, §4 SiluAndMul, §5 parallel Linear family,
 *         §6 vocab-parallel Embedding/LMHead, §7 attention, §8 assembly.
 *
 * Tensor parallelism is a weight LAYOUT on one device: `tp` shards are
 * slices of the same buffer; shard partial sums are reduced and logit
 * slices concatenated inside the kernels, with no collective.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless the parameter says "host".  The
 *     caller allocates and owns every buffer; the library keeps no pointer
 *     after the call returns.
 *   - Every tensor is dense row-major with the shape given; `dtype` is
 *     QW_BF16 or QW_F32 and applies to all floating-point tensors of the
 *     call except those documented as float (fp32) always.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronise.  Arguments are checked on the
 *     host before any launch; a failed check launches nothing.
 *   - The return value is a qw_status.  qw_last_error_string() describes the
 *     last failure on the calling thread.
 *   - A size of zero tokens is a valid no-op and returns QW_OK.
 *   - Workspaces (qw_attention_decode, qw_lm_head; sizes from the
 *     *_workspace_size queries) begin with 64 KiB of completion counters
 *     followed by scratch.  Zero-fill a workspace once when it is allocated;
 *     every call leaves the counters at zero again, so one workspace serves
 *     successive calls on one stream.  Calls that may run concurrently need
 *     separate workspaces.
 *   - One CUDA device per process: kernel attributes (shared-memory limits)
 *     are set once, on the device current at the first call.  Replicas on
 *     several GPUs run as one process each.
 *   - Environment switches, read on the host: QW_NO_PDL=1 launches every
 *     kernel without programmatic dependent launch (read once per process);
 *     QW_TC_PERSISTENT=1 runs many-token GEMMs on the persistent tensor-core
 *     kernel (two TMEM accumulators, one CTA per SM) instead of one CTA per
 *     output tile (read at each call; the outputs are bit-identical).
 *   - Device-side data errors (token id outside [0, V), position outside the
 *     RoPE table, slot outside the cache) do not fail the call: the affected
 *     row is zero (embedding, q) or not written (cache), and, when the
 *     caller passes a non-NULL `err_count` (device int32), it is incremented
 *     once per affected token.
 */
#ifndef QW_H
#define QW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QW_OK = 0,
  QW_ERR_INVALID_ARG = 1, /* null or misaligned pointer, negative size, bad enum */
  QW_ERR_SHAPE = 2,       /* a divisibility or size rule below is broken */
  QW_ERR_DTYPE = 3,       /* dtype not supported by this entry point */
  QW_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  QW_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (see qw_device_error) */
  QW_ERR_WORKSPACE = 6    /* workspace pointer missing or too small */
} qw_status;

typedef enum { QW_BF16 = 0, QW_F32 = 1 } qw_dtype;

typedef enum {
  QW_GEMM_COLUMN = 0,     /* W cut along the output dim ([TP] §3, tp_dim = 0) */
  QW_GEMM_ROW_REDUCE = 1  /* W cut along the input dim, shard partials summed ([TP] §3, tp_dim = 1) */
} qw_gemm_mode;

typedef enum {
  QW_EPI_NONE = 0,
  QW_EPI_SILU_MUL = 1     /* fused SiluAndMul on a merged gate_up output ([SK] §4) */
} qw_epilogue;

/* Version of this ABI (increments on any signature change); this is version 9. */
int qw_abi_version(void);

/* Description of the last failure on the calling thread ("" if none). */
const char* qw_last_error_string(void);

/*
 * Synchronises `stream`, then reports and clears the device-side error words.
 * Bounded waits inside the tensor-core and decode kernels set them when they
 * give up (a wait that should never time out; it exists so that a broken
 * pipeline returns instead of hanging the GPU): QW_ERR_TIMEOUT.  Decode
 * attention also records a context_lens entry larger than the max_context of
 * its call (the keys past max_context were not read, so that output is
 * wrong): QW_ERR_INVALID_ARG.  Returns QW_OK, QW_ERR_TIMEOUT or
 * QW_ERR_INVALID_ARG (QW_ERR_CUDA if the synchronisation fails).
 */
int qw_device_error(void* stream);

/*
 * Vocab-parallel embedding ([VH] §3, [VPE], [SK] §6).
 * For each token t and each shard r of `tp` (rows [r*V/tp, (r+1)*V/tp) of
 * the table): mask = id in the shard's range; local = mask * (id - start);
 * row = mask ? W_r[local] : 0; out[t] = sum over shards (the all_reduce).
 *   ids      int64 [T]
 *   table    dtype [V, H]   (shard r = row block r; the layout of tp stacked shards)
 *   out      dtype [T, H]
 *   err_count int32 [1] or NULL: +1 per id outside [0, V) (its row is zero)
 * Rules: V % tp == 0 (else QW_ERR_SHAPE); H * sizeof(dtype) % 16 == 0 and
 * table/out 16-byte aligned (else QW_ERR_INVALID_ARG).
 */
int qw_embed_vocab(const int64_t* ids, int64_t T, const void* table, int64_t V, int64_t H, int tp,
                   void* out, int32_t* err_count, int dtype, void* stream);

/*
 * Fused residual add + RMSNorm ([SK] §2 rms_forward / add_rms_forward, §1).
 * residual_in == NULL (first layer): s = x.  Otherwise s = round(x + residual_in).
 * residual_out (may alias residual_in, may be NULL) <- s;
 * y = round(s * rsqrt(mean(s^2) + eps) * gamma), computed in fp32.
 *   x, residual_in, residual_out, y : dtype [T, H];  gamma : dtype [H]
 * Rules: H * sizeof(dtype) % 16 == 0, H <= 4096 (bf16) or 2048 (f32),
 * 16-byte aligned pointers.  y must not alias x or residual_in.
 */
int qw_add_rmsnorm(const void* x, const void* residual_in, void* residual_out, const void* gamma,
                   float eps, int64_t T, int64_t H, void* y, int dtype, void* stream);

/*
 * RoPE cos/sin table on the HOST ([SK] §3): host_out float [max_position, rotary_dim]
 * with row p = [cos(p*f_0) .. cos(p*f_{d/2-1}), sin(p*f_0) .. sin(p*f_{d/2-1})],
 * f_i = fp32(1 / theta^(2i/d)), each angle the fp32 product p*f_i, cos/sin
 * rounded to fp32.  rotary_dim must be even and > 0.  Runs on the host only.
 */
int qw_rope_cos_sin_table(float* host_out, int64_t max_position, int rotary_dim, double theta);

/*
 * Per-head QK-RMSNorm, RoPE on q and k, KV-cache store ([SK] §8 ①, §3, §7.1).
 *   qkv       dtype [T, tp * (nh/tp + 2*nkv/tp) * hd]: the merged QKV output,
 *             shard r's block = [q_r | k_r | v_r] ([SK] §5 QKVParallelLinear)
 *   positions int64 [T];  cos_sin float [max_position, hd] (qw_rope_cos_sin_table)
 *   q_gamma, k_gamma dtype [hd]
 *   slot_mapping int64 [T]: cache row of each token, -1 = do not store
 *   k_cache, v_cache dtype [num_slots, nkv, hd] (kv head g = shard g/(nkv/tp))
 *   q_out     dtype [T, nh, hd]
 * Per q head: q = round(rmsnorm(q) * q_gamma); q_out = round(rope(q)).
 * Per kv head: k likewise with k_gamma, stored with the raw v to the cache.
 * Rules: nh % tp == 0, nkv % tp == 0, hd even and <= 256.
 */
int qw_qkv_norm_rope_store_kv(const void* qkv, int64_t T, int n_heads, int n_kv_heads, int head_dim,
                              int tp, const int64_t* positions, const float* cos_sin,
                              int64_t max_position, const void* q_gamma, const void* k_gamma, float eps,
                              const int64_t* slot_mapping, void* k_cache, void* v_cache, int64_t num_slots,
                              void* q_out, int32_t* err_count, int dtype, void* stream);

/*
 * A row-parallel Linear whose output joins the residual stream, followed by
 * the next RMSNorm ([SK] §1-§2 add_rms_forward, [TP] §3 Y = sum_r X_r W_r^T):
 * qw_gemm (ROW_REDUCE) then qw_add_rmsnorm, in one launch for many tokens
 * (prefill o_proj and down_proj):
 *   residual <- round(round(A W^T) + residual)            (in place)
 *   y        <- round(residual * rsqrt(mean(residual^2) + eps) * gamma)
 *   A bf16 [M, K];  W bf16 [tp, N, K/tp] (shard r = input columns r);
 *   residual bf16 [M, N] (read and written);  gamma bf16 [N];  y bf16 [M, N]
 * The N/256 column tiles of a 128-row block run as one thread-block cluster
 * and add their rows' sums of squares in tile order over distributed shared
 * memory.  Rounding points as qw_gemm + qw_add_rmsnorm; the sum of squares is
 * accumulated in another order (fp32), so y may differ from that pair of
 * calls by one bf16 step where it lies next to a rounding midpoint.
 * Rules: bf16; N a multiple of 256 up to 2048; K % tp == 0, (K/tp) % 8 == 0;
 * 16-byte aligned pointers; y must not alias residual.  Errors: QW_ERR_DTYPE,
 * QW_ERR_SHAPE, QW_ERR_INVALID_ARG.
 */
int qw_gemm_add_rmsnorm(const void* A, const void* W, int64_t M, int64_t N, int64_t K, int tp, void* residual,
                        const void* gamma, float eps, void* y, int dtype, void* stream);

/*
 * The merged QKV projection with its per-head QK-RMSNorm, RoPE and KV-cache
 * store as the GEMM's epilogue ([SK] §5 QKVParallelLinear, §8 ①, §3, §7.1):
 * qw_gemm (COLUMN) of A [T, H] by W followed by qw_qkv_norm_rope_store_kv,
 * with the same results bit for bit, except that the QKV output never goes
 * to memory.  For many tokens (prefill): every token row runs on a 128-row
 * tensor-core tile.
 *   A bf16 [T, H];  W bf16 [tp * (nh/tp + 2*nkv/tp) * 128, H], shard r's rows
 *   [q_r; k_r; v_r] (the layout of qw_qkv_norm_rope_store_kv's qkv columns);
 *   positions, cos_sin, max_position, q_gamma, k_gamma, eps, slot_mapping,
 *   k_cache, v_cache, num_slots, q_out, err_count: as for
 *   qw_qkv_norm_rope_store_kv (head_dim 128).
 * Rules: bf16; head_dim 128; tp divides nh and nkv; (nh + 2*nkv)/tp even (a
 * 256-column tile holds two whole heads of one shard); H % 8 == 0; 16-byte
 * aligned pointers.  Errors: QW_ERR_DTYPE, QW_ERR_SHAPE, QW_ERR_INVALID_ARG.
 */
int qw_qkv_gemm_norm_rope_store_kv(const void* A, const void* W, int64_t T, int64_t H, int n_heads, int n_kv_heads,
                                   int head_dim, int tp, const int64_t* positions, const float* cos_sin,
                                   int64_t max_position, const void* q_gamma, const void* k_gamma, float eps,
                                   const int64_t* slot_mapping, void* k_cache, void* v_cache, int64_t num_slots,
                                   void* q_out, int32_t* err_count, int dtype, void* stream);

/*
 * Causal varlen GQA attention for prefill (flash_attn_varlen_func with
 * causal=True, [SK] §7.2).
 *   q   dtype [Tq, nh, hd], sequences packed by cu_seqlens_q (int32 [n_seqs+1])
 *   k,v dtype [kv_rows, nkv, hd] (16-byte aligned): key j of sequence s is row
 *       seq_base[s] + j when seq_base (int32 [n_seqs]) is given (keys read
 *       from the KV cache), else row cu_seqlens_k[s] + j (packed keys); every
 *       row read must be < kv_rows (the bf16 head_dim-128 path reads k and v
 *       through TMA tensor maps bounded by kv_rows).
 *   cu_seqlens_k int32 [n_seqs+1]: Lk_s = cu_seqlens_k[s+1] - cu_seqlens_k[s] >= Lq_s;
 *       query i of sequence s sits at key position Lk_s - Lq_s + i and sees
 *       keys 0 .. that position.
 *   out dtype [Tq, nh, hd];  q head h reads kv head h / (nh / nkv).
 *   max_seqlen_q: upper bound of Lq_s (sizes the grid).
 * Rules: nh % nkv == 0; hd == 128 (bf16, tensor-core path) or hd <= 64 (bf16 or
 * f32, CUDA-core path).
 */
int qw_attention_prefill(const void* q, const void* k, const void* v, int64_t kv_rows,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* seq_base,
                         int n_seqs, int max_seqlen_q, int n_heads, int n_kv_heads, int head_dim, float scale,
                         void* out, int dtype, void* stream);

/*
 * Decode attention over the KV cache (flash_attn_with_kvcache, [SK] §7.2):
 * one new query token per sequence, sees cache rows
 * seq_base[b] .. seq_base[b] + context_lens[b] - 1 (the token just stored included).
 *   q   dtype [B, nh, hd];  k_cache, v_cache dtype [num_slots, nkv, hd] (16-byte aligned)
 *   context_lens, seq_base int32 [B];  max_context >= every context_lens[b]
 *   (it sizes the split of the keys over CTAs; max_context 0 means every
 *   sequence is empty and gets a zero output; an entry above max_context is
 *   not an argument error the host can see, so the kernel records it for
 *   qw_device_error, which returns QW_ERR_INVALID_ARG);
 *   every cache row read, seq_base[b] .. seq_base[b] + context_lens[b] - 1, < num_slots
 *   out dtype [B, nh, hd]
 *   workspace: device scratch of qw_attention_decode_workspace_size(...) bytes
 *   (split-KV partial results); may be NULL only when that size is 0.  The
 *   first 64 KiB are completion counters: zero before the first call, and
 *   every call leaves them zero, including a call whose bounded wait gave up
 *   (every CTA still runs to its end and counts itself in).
 *   flags: 0, or QW_DECODE_HISTORY_READY (bf16, hd 128).  With that flag the
 *   caller states that context_lens, seq_base and every cache row the call
 *   reads except each sequence's last (position context_lens[b] - 1) were
 *   complete before the kernel enqueued just before this call started, and
 *   that this kernel writes at most q and those last rows (a decode step's
 *   QK-norm + RoPE + KV store).  The kernel then reads the lengths and starts
 *   copying the earlier rows before it waits for that kernel (programmatic
 *   dependent launch).  Without it nothing is read before the wait.
 * Rules: nh % nkv == 0; hd == 128 with nh/nkv in {1, 2, 4, 8} (split-KV path),
 * or hd <= 64 (one warp per (sequence, q head), no workspace); bf16 or f32;
 * unknown flags: QW_ERR_INVALID_ARG.
 */
#define QW_DECODE_HISTORY_READY 1
int qw_attention_decode(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                        const int32_t* context_lens, const int32_t* seq_base, int B, int max_context,
                        int n_heads, int n_kv_heads, int head_dim, float scale, void* out,
                        void* workspace, size_t workspace_bytes, int dtype, int flags, void* stream);
size_t qw_attention_decode_workspace_size(int B, int max_context, int n_heads, int head_dim);

/*
 * Paged KV cache ([SK] §7.2; nano-vllm's block_table with block_size 256):
 * key position p of sequence s is cache row
 *   block_table[s * max_blocks + p / block_size] * block_size + p % block_size.
 * The caller owns block_table (int32 [n_seqs, max_blocks], device) and keeps
 * every entry a sequence uses a valid block: rows outside [0, num_slots) read
 * as zeros.  Both entry points are bf16 with head_dim 128.
 *
 * qw_attention_decode_paged: qw_attention_decode with the block table in place
 *   of seq_base.  block_size a multiple of 64; max_context <= max_blocks *
 *   block_size.  flags: 0 or QW_DECODE_HISTORY_READY (the block table then
 *   counts among the inputs complete before the previous kernel started).
 * qw_attention_prefill_paged: causal prefill attention with every key read
 *   from the cache through the block table, the prefix-cache prefill: query i
 *   of sequence s (Lq_s = cu_seqlens_q[s+1] - cu_seqlens_q[s] new tokens) sits
 *   at key position Lk_s - Lq_s + i, Lk_s = cu_seqlens_k[s+1] - cu_seqlens_k[s]
 *   keys cached (new tokens' k/v stored first).  block_size a multiple of 128.
 * Errors: QW_ERR_DTYPE, QW_ERR_SHAPE (head_dim, group, block_size,
 * max_context), QW_ERR_INVALID_ARG (null or misaligned pointers, flags),
 * QW_ERR_WORKSPACE (decode).
 */
int qw_attention_decode_paged(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                              const int32_t* context_lens, const int32_t* block_table, int max_blocks, int block_size,
                              int B, int max_context, int n_heads, int n_kv_heads, int head_dim, float scale,
                              void* out, void* workspace, size_t workspace_bytes, int dtype, int flags, void* stream);
int qw_attention_prefill_paged(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* block_table,
                               int max_blocks, int block_size, int n_seqs, int max_seqlen_q, int n_heads,
                               int n_kv_heads, int head_dim, float scale, void* out, int dtype, void* stream);

/*
 * Decode step's QK-RMSNorm + RoPE + KV-cache store ([SK] §3, §7.1, §8) and
 * decode attention ([SK] §7.2) in one launch: qw_qkv_norm_rope_store_kv on
 * one token per sequence followed by qw_attention_decode, without the q_out
 * round trip.
 *   qkv bf16 [B, tp * (nh/tp + 2*nkv/tp) * 128]: the merged QKV output, shard r
 *       holding [q_r; k_r; v_r] (as for qw_qkv_norm_rope_store_kv);
 *   positions int64 [B], cos_sin, max_position, q_gamma, k_gamma, eps,
 *       slot_mapping int64 [B], err_count: as for qw_qkv_norm_rope_store_kv;
 *   k_cache, v_cache bf16 [num_slots, nkv, 128] (16-byte aligned);
 *   context_lens, seq_base, max_context, scale, out, workspace, flags: as for
 *       qw_attention_decode (workspace from qw_attention_decode_workspace_size);
 *       with QW_DECODE_HISTORY_READY the caller also states that positions were
 *       complete before the previous kernel started, and the kernel reads them,
 *       the gammas and cos_sin before it waits.
 * Sequence b's key positions 0 .. context_lens[b] - 1 sit at cache rows
 * seq_base[b] + position, and this step's k and v are the ones at position
 * context_lens[b] - 1: slot_mapping[b] must be seq_base[b] + context_lens[b]
 * - 1, or -1 for a sequence whose k/v is not stored (then context_lens[b] must
 * not count it).  A sequence with context_lens[b] = 0 stores nothing and gets
 * a zero output.  Rules: bf16, head_dim 128, nh % nkv == 0 with group 1/2/4/8,
 * tp divides nh and nkv.
 */
int qw_attention_decode_rope(const void* qkv, int n_heads, int n_kv_heads, int head_dim, int tp,
                             const int64_t* positions, const float* cos_sin, int64_t max_position,
                             const void* q_gamma, const void* k_gamma, float eps, const int64_t* slot_mapping,
                             void* k_cache, void* v_cache, int64_t num_slots, int32_t* err_count,
                             const int32_t* context_lens, const int32_t* seq_base, int B, int max_context,
                             float scale, void* out, void* workspace, size_t workspace_bytes, int dtype, int flags,
                             void* stream);

/*
 * Decode attention that needs no workspace from the caller.  The pages have
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory themselves, such as a plugin that a host framework hands
 * only input and output pointers (the framework owns the allocator), or a
 * serving loop that sizes all device memory at start-up and forbids any
 * later allocation.
 *
 * Same arguments, semantics and results as qw_attention_decode, minus the
 * workspace: the split-KV partial results go to one fixed array of
 * qw_attention_decode_static_scratch_bytes() bytes (2 MiB) that lives in the
 * library's device image; every GPU that loads the library holds it until
 * the process exits.  A batch whose split-KV scratch
 * (qw_attention_decode_workspace_size) exceeds that size is rejected with
 * QW_ERR_WORKSPACE and nothing is launched.  The call makes no allocation
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * The first call on a device looks up the array's device address on that
 * device (the caller's current device), once; make that first call before
 * any stream capture.
 *
 * All calls share the one array and it keeps whatever the last call left in
 * it.  Its first 64 KiB are completion counters that must be zero when a
 * call starts: the array is zero when the library is loaded and every call
 * leaves its counters at zero; the rest of the array needs no clearing,
 * because every value a call reads there was written earlier in the same
 * call.  A call whose bounded wait gave up (qw_device_error returns
 * QW_ERR_TIMEOUT) still runs every CTA to its end, so it too leaves the
 * counters at zero; only its output is invalid.  Calls that can run at the
 * same time on the GPU (on two streams, or from two host threads) race on
 * the array and give wrong results: keep them on one stream.  Each process
 * has its own copy of the array.  Its results are bit-identical to
 * qw_attention_decode's with a workspace (same kernels, same partition).
 */
int qw_attention_decode_static(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                               const int32_t* context_lens, const int32_t* seq_base, int B, int max_context,
                               int n_heads, int n_kv_heads, int head_dim, float scale, void* out, int dtype,
                               void* stream);
size_t qw_attention_decode_static_scratch_bytes(void);

/*
 * Self-test of the failure path: launches one thread that waits on an
 * mbarrier that nothing completes.  The wait is bounded like every wait of
 * the tensor-core kernels (2 s of %globaltimer); when it gives up it records
 * code 0x100 in the tensor-core error word and the kernel returns.  The next
 * qw_device_error on the stream then returns QW_ERR_TIMEOUT and clears the
 * word.  No fault, no trap; the context stays usable.  It has no counterpart in
 * the cited sources.  Errors: QW_ERR_CUDA if the launch fails.
 */
int qw_selftest_wait_timeout(void* stream);

/*
 * Linear layer C = A W^T with the tensor-parallel layouts of [TP] §3 / [SK] §5.
 *   A dtype [M, K]
 *   QW_GEMM_COLUMN:     W dtype [N, K] (tp shards stacked along N; shard r = rows
 *                       [r*N/tp, (r+1)*N/tp)); C[M, N] = A W^T.
 *     with QW_EPI_SILU_MUL: N = 2*I and shard r's rows are [gate_r (I/tp) ; up_r (I/tp)]
 *                       ([SK] §5 MergedColumnParallelLinear); C is [M, I] with
 *                       C[:, r*I/tp + j] = silu(G[:, j]) * U[:, j] of shard r.
 *   QW_GEMM_ROW_REDUCE: W dtype [tp, N, K/tp] (shard r holds input columns
 *                       [r*K/tp, (r+1)*K/tp)); C[M, N] = sum_r A[:, shard r] W_r^T,
 *                       accumulated in fp32 across shards (the all_reduce), rounded once.
 *   workspace: unused (pass NULL, 0); qw_gemm_workspace_size returns 0.  With
 *   few tokens (<= 64) the K range is split either over the 8 warps of a CTA
 *   that owns 16 weight rows (K/tp % 32 == 0; up to 8 tokens the rows are
 *   bulk-copied into shared memory ahead of the programmatic wait) or over a
 *   thread-block cluster; the partial sums are added in shared memory, in a
 *   fixed order.
 * Rules (bf16): K % 8 == 0, K/tp % 8 == 0 (row), N % 16 == 0 (N/2/tp % 8 == 0 for
 * SILU_MUL), A/W/C 16-byte aligned.  f32 runs on CUDA cores (exact fp32 FMA).
 */
int qw_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K, int tp, int mode,
            int epilogue, void* workspace, size_t workspace_bytes, int dtype, void* stream);
size_t qw_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int tp, int mode, int epilogue, int dtype);

/*
 * SiluAndMul on a merged gate_up output ([SK] §4, [TP] §4.2).
 *   x dtype [T, 2*I] with shard r's block [gate_r (I/tp) | up_r (I/tp)];
 *   out dtype [T, I], out[:, r*I/tp + j] = round(silu(gate_r[j]) * up_r[j]).
 * Rules: I % tp == 0, (I/tp) * sizeof(dtype) % 16 == 0.
 */
int qw_silu_mul(const void* x, void* out, int64_t T, int64_t I, int tp, int dtype, void* stream);

/*
 * Fused add + RMSNorm and Linear for few tokens (decode): the
 * input_layernorm / post_attention_layernorm of Qwen3DecoderLayer feeding
 * the QKV or gate_up projection ([SK] §1, §2, §5).  Same arithmetic and
 * rounding points as qw_add_rmsnorm followed by qw_gemm (column layout):
 *   s = x + residual_in (rounded to bf16; s = x when residual_in is NULL)
 *   residual_out = s (if not NULL); y = RMSNorm(s) * gamma (rounded); C = y W^T
 *   x, residual_in, residual_out bf16 [M, K];  gamma bf16 [K]
 *   W bf16 [N, K] (column layout: tp shards stacked along N);  C bf16 [M, N],
 *   or [M, N/2] with QW_EPI_SILU_MUL (gate_up, as qw_gemm)
 * Rules: bf16; 0 <= M <= 16; K % 32 == 0, N % 16 == 0 and qw_gemm's shard
 * rules; M * (K + 8) * 2 <= 211 KiB (the normed rows live in shared memory);
 * 16-byte aligned pointers; residual_out must not alias x or residual_in
 * (every CTA reads them while one writes it).  Otherwise QW_ERR_SHAPE /
 * QW_ERR_INVALID_ARG.
 */
int qw_add_rmsnorm_gemm(const void* x, const void* residual_in, void* residual_out, const void* gamma, float eps,
                        const void* W, void* C, int64_t M, int64_t N, int64_t K, int tp, int epilogue, int dtype,
                        void* stream);

/*
 * Vocab-parallel lm_head with the tied table ([VH] §4, [SK] §6, §8) and greedy
 * sampling.
 *   hidden    dtype [T, H]
 *   last_idx  int32 [n_out] or NULL.  Prefill: row last_idx[i] of hidden is
 *             projected (cu_seqlens_q[1:] - 1).  NULL: rows 0 .. n_out-1.
 *   table     dtype [V, H]  (shard r = vocab rows [r*V/tp, (r+1)*V/tp); its logit
 *             slice lands at columns [r*V/tp, (r+1)*V/tp): the gather + cat)
 *   logits    dtype [n_out, V]
 *   next_tokens int64 [n_out] or NULL: argmax over each logits row, lowest index on ties
 *   workspace: qw_lm_head_workspace_size(...) bytes.
 * Rules: V % tp == 0, V % 16 == 0, H % 8 == 0.
 */
int qw_lm_head(const void* hidden, int64_t T, const int32_t* last_idx, int64_t n_out, const void* table,
               int64_t V, int64_t H, int tp, void* logits, int64_t* next_tokens, void* workspace,
               size_t workspace_bytes, int dtype, void* stream);
size_t qw_lm_head_workspace_size(int64_t n_out, int64_t V, int64_t H, int tp, int dtype);

/* Greedy argmax over rows of logits dtype [M, V] -> int64 [M], lowest index on ties. */
int qw_argmax(const void* logits, int64_t M, int64_t V, int64_t* out, int dtype, void* stream);

/*
 * Temperature / top-p sampling of one token per row: the Sampler that
 * nano-vllm compiles with RMSNorm, RoPE and SiluAndMul ([SK] §3).  The pages
 * give no semantics; this is the reading implemented:
 *   temperature[b] <= 0 (or NaN): greedy, argmax with the lowest index on ties
 *   (top_p and uniforms of that row are not read);
 *   otherwise the token is drawn from softmax(logits[b] / T) restricted to the
 *   nucleus: the row's distinct logit values are taken from the largest down
 *   until their softmax mass reaches top_p[b] of the row's mass, and every
 *   token whose logit is at least the last value taken is kept (tokens tied
 *   at the boundary are all kept; top_p outside (0, 1] keeps the whole row).
 *   The draw is the Gumbel-max identity: argmax over the nucleus of
 *   logits / T - log(-log u), lowest index on ties.
 *   logits      bf16 [B, V], finite, 16-byte aligned
 *   temperature float [B], top_p float [B] (device)
 *   uniforms    float [B, V] (device, 16-byte aligned): the random numbers of
 *               the draw, each in (0, 1) (clamped to [2^-24, 1 - 2^-24]);
 *               supplied by the caller so that draws are reproducible
 *   out         int64 [B]
 *   workspace:  qw_sample_workspace_size(B, V) bytes, 16-byte aligned, zero
 *               when first used; every call leaves it ready for the next
 *               (calls that may run concurrently need separate workspaces).
 * Three launches; results do not depend on timing (fixed reduction orders).
 * Rules: bf16 (else QW_ERR_DTYPE); V a positive multiple of 8 below 2^30;
 * B <= 16384.  Errors: QW_ERR_INVALID_ARG, QW_ERR_SHAPE, QW_ERR_WORKSPACE.
 */
int qw_sample(const void* logits, int64_t B, int64_t V, const float* temperature, const float* top_p,
              const float* uniforms, int64_t* out, void* workspace, size_t workspace_bytes, int dtype,
              void* stream);
size_t qw_sample_workspace_size(int64_t B, int64_t V);

/*
 * One decode step of every decoder layer in one persistent kernel: for each
 * layer, in the order of Qwen3DecoderLayer.forward ([SK] §1, §8):
 *   add + RMSNorm (input_layernorm) -> QKV (column layout) -> QK-RMSNorm,
 *   RoPE, KV-cache store -> decode attention over the cache -> o_proj (row
 *   layout, shard sums) -> add + RMSNorm (post_attention_layernorm) ->
 *   gate_up (column) + SiluAndMul -> down (row)
 * and then the final add + RMSNorm.  Same arithmetic, layouts and rounding
 * points as the per-operation entry points above; it exists because a
 * decode batch of a few tokens leaves each operation far too small to fill
 * the GPU on its own.
 *   layers   host array of n_layers qw_decode_layer records (pointers into
 *            device memory; the layouts of qw_gemm / qw_qkv_norm_rope_store_kv),
 *            read during the call; the K/V caches 16-byte aligned
 *   x        bf16 [B, H]: the embedding of the B new tokens (layer 0 input)
 *   positions, slot_mapping int64 [B]; context_lens, seq_base int32 [B]:
 *            as for qw_qkv_norm_rope_store_kv and qw_attention_decode (the new
 *            token's k/v go to slot_mapping[b], which must be
 *            seq_base[b] + context_lens[b] - 1; max_context >= every
 *            context_lens[b])
 *   cos_sin  fp32 [max_position, head_dim] (qw_rope_cos_sin_table)
 *   final_norm bf16 [H];  out bf16 [B, H]: final normed hidden (lm_head input)
 *   err_count int32 [1] or NULL: +1 per position or slot out of range
 *   workspace: qw_decode_layers_workspace_size(...) bytes, 16-byte aligned,
 *            zero when first used.  Every call leaves its first 64 KiB (grid
 *            barrier, counters) as a following call needs them; after a call
 *            that qw_device_error reports as timed out, zero it again.
 * Rules: bf16; 1 <= B <= 16; head_dim 128; nh/nkv in {1, 2, 4, 8}; nh, nkv
 * and I divisible by tp; H, nh*128/tp and I/tp multiples of 256;
 * n_layers <= 64.  Launched cooperatively with one CTA per SM: calls on
 * different streams must not overlap.  Errors: QW_ERR_SHAPE,
 * QW_ERR_INVALID_ARG, QW_ERR_WORKSPACE, QW_ERR_CUDA.
 */
typedef struct qw_decode_layer {
  const void* input_layernorm;           /* bf16 [H] */
  const void* qkv;                       /* bf16 [tp * (nh/tp + 2*nkv/tp) * hd, H] */
  const void* q_norm;                    /* bf16 [hd] */
  const void* k_norm;                    /* bf16 [hd] */
  const void* o_proj;                    /* bf16 [tp, H, nh/tp * hd] */
  const void* post_attention_layernorm;  /* bf16 [H] */
  const void* gate_up;                   /* bf16 [tp * 2*I/tp, H] */
  const void* down;                      /* bf16 [tp, H, I/tp] */
  void* k_cache;                         /* bf16 [num_slots, nkv, hd] */
  void* v_cache;                         /* bf16 [num_slots, nkv, hd] */
} qw_decode_layer;

int qw_decode_layers(const qw_decode_layer* layers, int n_layers, const void* x, const int64_t* positions,
                     const int64_t* slot_mapping, const int32_t* context_lens, const int32_t* seq_base, int B,
                     int max_context, int H, int n_heads, int n_kv_heads, int head_dim, int intermediate, int tp,
                     const float* cos_sin, int64_t max_position, int64_t num_slots, float eps, float scale,
                     const void* final_norm, void* out, int32_t* err_count, void* workspace,
                     size_t workspace_bytes, void* stream);
size_t qw_decode_layers_workspace_size(int n_layers, int B, int H, int n_heads, int n_kv_heads, int head_dim,
                                       int intermediate, int tp, int max_context);

#ifdef __cplusplus
}
#endif

#endif /* QW_H */
