/*
 * attn.h - C ABI of libattn: fused scaled-dot-product attention, forward and backward,
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (forward): for every batch b and query head h, with kv head
 * kvh = h / (Hq / Hkv) and L = the valid key length of (b, kvh),
 *
 *     S    = scale * Q[b, :, h, :] . K[b, :L, kvh, :]^T          (Sq x L)
 *     S_ij = -inf where causal and j > i + (L - Sq)               (bottom-right aligned)
 *     O    = softmax_rows(S) . V[b, :L, kvh, :]                  (Sq x D)
 *     LSE  = log(sum_j exp(S_ij))   (natural log, fp32)
 *
 * computed without materialising S: an online softmax over K/V tiles with a running
 * max and sum ("xtrain evolution.md", infra table row T14: fused flash attention,
 * online softmax tiled over KV, no N x N scores). Query heads share kv heads in groups
 * of Hq / Hkv (row T15: true GQA, dst = kvh * group + r). Keys at or past the valid
 * length are padding and never influence a result ("LingBot full-pipeline analysis
 * report", section "same-GPU FA2/FA3 hardware comparison": the FP64 reference uses only
 * the cu_seqlens-valid K/V). A query row with no visible key gets O = 0, LSE = -inf.
 *
 * The backward (row T14: recompute the scores, D = sum(dO * O) simplifies the softmax
 * Jacobian) gives dQ, dK, dV of sum(O * dO); kv-head gradients are the sum over the
 * query heads of the group in a fixed order (row T15: deterministic in-group sum, no
 * atomics). Results are bitwise reproducible run to run for identical inputs.
 *
 * Layout (all contiguous, row-major, D innermost; the pages' token-major [tokens, H, D]
 * with a batch dimension in front):
 *     q, o, dout, dq : [B, Sq,  Hq,  D]
 *     k, v, dk, dv   : [B, Skv, Hkv, D]
 *     lse            : [B, Hq, Sq]  fp32
 *     kv_lens        : [B, Hkv]     int32, device memory, or NULL (= every length Skv)
 * Element type: ATTN_BF16 (bfloat16) or ATTN_F32 (float) for q, k, v, o, dout, dq, dk,
 * dv; lse is always fp32; accumulation is always fp32. Outputs are rounded to the
 * element type with round-to-nearest-even.
 *
 * Ownership and streams: every pointer is a device pointer owned by the caller; the
 * library never allocates, frees or retains one. Calls are asynchronous on `stream`
 * (NULL = the legacy default stream) and never modify their inputs. The backward needs
 * a caller-provided device workspace of attn_bwd_workspace_size() bytes.
 *
 * Errors: argument checks are synchronous, on the host, before anything is launched;
 * a failed check returns a negative status and launches nothing. Values that live in
 * device memory (kv_lens) cannot be checked on the host: the kernels clamp them to
 * [0, Skv] and record the fact in a device error word, which attn_peek_device_error()
 * reads. Kernels that wait on barriers bound every wait; a wait that runs out records
 * ATTN_DEVERR_TIMEOUT and the kernel returns instead of hanging.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (binary-compatible with cudaStream_t / CUstream). */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_BF16 = 0, /* bfloat16 inputs and outputs */
  ATTN_F32 = 1   /* float inputs and outputs */
} attn_dtype_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* a null/misaligned pointer, a bad size, a non-finite scale */
  ATTN_ERR_UNSUPPORTED = -2, /* a valid request this library does not implement (e.g. D) */
  ATTN_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  ATTN_ERR_TIMEOUT = -4,     /* a device-side bounded wait ran out (see the error word) */
  ATTN_ERR_WORKSPACE = -5    /* the backward workspace is missing or too small */
} attn_status_t;

/* Bits of the device error word. */
#define ATTN_DEVERR_KVLEN 0x1u   /* a kv_lens entry was outside [0, Skv]; it was clamped */
#define ATTN_DEVERR_TIMEOUT 0x2u /* a bounded barrier wait ran out; outputs are invalid */
#define ATTN_DEVERR_LAYOUT 0x4u  /* a kernel's shared memory was not 1024-byte aligned, which
                                    its swizzled tiles need; it computed nothing, outputs are
                                    invalid */
#define ATTN_DEVERR_PAGE 0x8u    /* a block-table entry that a paged forward needed was not a
                                    page of the pool; page 0 was read instead, outputs are
                                    invalid */

/*
 * Forward. q, k, v: inputs; o: output [B, Sq, Hq, D]; lse: output [B, Hq, Sq] fp32.
 * B, Sq >= 0 (0 = nothing to do); Hq, Hkv >= 1 with Hq % Hkv == 0; Skv >= 0 (0 = every
 * row empty); D in {64, 128} (else ATTN_ERR_UNSUPPORTED); scale finite; causal 0 or 1.
 * Pointers to q, k, v, o must be 16-byte aligned; lse and kv_lens 4-byte aligned.
 */
ATTN_API attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                       int causal, const int32_t* kv_lens, attn_dtype_t dtype,
                       attn_stream_t stream);

/*
 * Backward. q, k, v, o, lse: the forward's inputs and outputs; dout: the gradient of O
 * [B, Sq, Hq, D]; dq, dk, dv: outputs (dk, dv are zero at keys past the valid length).
 * The same size, alignment and kv_lens rules as attn_fwd; in addition dout, dq, dk,
 * dv must be 16-byte aligned and `workspace` must hold at least
 * attn_bwd_workspace_size(...) bytes of device memory, 256-byte aligned, for the call's
 * exclusive use until the stream reaches the end of the call (ATTN_ERR_WORKSPACE
 * otherwise). The workspace holds delta = rowsum(dO * O) [B, Hq, Sq] fp32 and, when
 * attn_bwd_workspace_size() says so, fp32 partial dK/dV of runs of query heads.
 */
ATTN_API attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                       int causal, const int32_t* kv_lens, attn_dtype_t dtype,
                       void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * Paged forward: attention over a K/V cache kept in fixed-size pages, read through a
 * per-sequence block table instead of first gathering the pages into contiguous K/V
 * ("LingBot full-pipeline analysis report", section "optimisation migration matrix v2",
 * row H1a_kv_gather_off: direct paged FA through the block table against gather + FA
 * varlen; the self-attention cache keeps a block table and per-sequence lengths,
 * section "layer-0 internal diagnosis v5").
 *     q, o             : [B, Sq, Hq, D] bf16
 *     k_pages, v_pages : [num_pages, page_size, Hkv, D] bf16, the key and value pools
 *     block_table      : [B, max_pages] int32, device memory: entry t of sequence b is the
 *                        page that holds its keys t * page_size .. (t + 1) * page_size - 1;
 *                        only entries of pages that hold valid keys are read
 *     seq_lens         : [B] int32, device memory: valid keys of each sequence, shared by
 *                        its kv heads; NULL = max_pages * page_size for every sequence
 *     lse              : [B, Hq, Sq] fp32
 * The result is attn_fwd on the gathered K/V [B, max_pages * page_size, Hkv, D] with
 * kv_lens[b][kvh] = seq_lens[b]: the same GQA, causal (bottom-right) and empty-row rules.
 * page_size must be a power of two of at least 16, num_pages and max_pages >= 1, dtype
 * ATTN_BF16 (else ATTN_ERR_UNSUPPORTED; the other checks are those of attn_fwd). A
 * seq_lens entry outside [0, max_pages * page_size] is clamped and flagged
 * (ATTN_DEVERR_KVLEN); a needed block-table entry outside [0, num_pages) is flagged
 * (ATTN_DEVERR_PAGE) and page 0 is read in its place. Pointers: q, k_pages, v_pages, o
 * 16-byte aligned; block_table, seq_lens, lse 4-byte aligned.
 */
ATTN_API attn_status_t attn_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                                      int num_pages, int page_size, int max_pages, int D,
                                      float scale, int causal, attn_dtype_t dtype,
                                      attn_stream_t stream);

/*
 * Split-KV forward, for short query blocks over long K/V: single-query decode ("xtrain
 * evolution.md", phase-3 milestone M2a: decode attention equals the last causal row of
 * the full computation) and a few query rows against a whole cache, where the per-rank
 * work is too short to fill the GPU (LingBot report, section "Attention effective-FLOP
 * utilisation curve (A0)": utilisation falls as the per-call work shrinks). Arguments,
 * layout, results and errors are those of attn_fwd, plus a workspace of
 * attn_fwd_splitkv_workspace_size() bytes of device memory (256-byte aligned, for the
 * call's exclusive use until the stream reaches its end; ATTN_ERR_WORKSPACE otherwise).
 * Each (batch, head, 128-row query block) is cut into ranges of key tiles processed as
 * separate work items; an item writes its normalised partial O and LSE (fp32) to the
 * workspace and a second kernel merges a row's ranges in range order (deterministic):
 * lse = log(sum_s exp(lse_s)), O = sum_s exp(lse_s - lse) O_s. When the problem already
 * has enough work items the call is exactly attn_fwd and the workspace is not touched.
 */
ATTN_API attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int B, int Hq, int Hkv, int Sq, int Skv,
                                        int D, float scale, int causal, const int32_t* kv_lens,
                                        attn_dtype_t dtype, void* workspace,
                                        size_t workspace_bytes, attn_stream_t stream);

/* Bytes of device workspace attn_fwd_splitkv needs for these sizes: 0 when it does not
 * split (fp32, or enough (batch, head, query block) items: at least 152), else
 * n * B * Hq * Sq * D * 4 bytes of partial O plus n * B * Hq * Sq * 4 bytes of partial LSE
 * (each rounded up to 256) for n key ranges per item. With T tiles of 128 keys and I
 * items, n is the count in 1 .. T / 4 (a range holds at least 4 tiles) that minimises a
 * model of the time, ceil(I * n / 152) rounds of 2 * ceil(T / n) + 6 half-tile steps,
 * then reduced to the number of ranges of ceil(T / n) tiles that cover T. A pure function
 * of the sizes. */
ATTN_API size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                                attn_dtype_t dtype);

/*
 * Forward on tensors in pinned host memory: attn_fwd's operation and results (bit for
 * bit), for callers whose activations live on the host. q, k, v, o, lse (and kv_lens,
 * if not NULL) are host pointers in attn_fwd's layouts, page-locked (cudaHostAlloc or
 * cudaHostRegister; other memory, including device memory, gives ATTN_ERR_INVALID_ARG).
 * The problem is computed in chunks of about a fifth of the kv heads (with their query
 * heads): the inputs of one chunk are copied in while the previous chunk is computed and
 * the one before it copied out, so the link and the GPU work at the same time.
 * `workspace`: device memory of attn_fwd_host_workspace_size() bytes, 256-byte aligned,
 * for the call's exclusive use until `stream` reaches the end of the call
 * (ATTN_ERR_WORKSPACE otherwise); it holds two chunks' inputs and outputs. The call is
 * asynchronous on `stream`: the copies wait for the work queued on `stream` before the
 * call, and work queued after it (or a synchronisation of `stream`) sees o and lse
 * written. The compute runs on `stream`, the copies on two streams of the library's own.
 * Argument errors are found before anything is queued. A CUDA error met while queueing the
 * chunks is returned as ATTN_ERR_CUDA after some chunks' copies may already be queued:
 * synchronize the device before reusing the workspace or the host buffers. Calls from
 * several threads are serialised while they queue their work. The other rules are
 * attn_fwd's.
 */
ATTN_API attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                       float scale, int causal, const int32_t* kv_lens, attn_dtype_t dtype,
                       void* workspace, size_t workspace_bytes, attn_stream_t stream);
ATTN_API size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                       attn_dtype_t dtype);

/* Bytes of device workspace attn_bwd needs for these sizes (0 for an empty problem):
 * delta [B, Hq, Sq] fp32, plus, for bf16 GQA problems with fewer than 256 (batch, kv
 * head, 128-key tile) work items, fp32 partial dK and dV [B, Skv, Hkv * P, D] that a
 * second kernel sums over each group in a fixed order. P, the number of parts each
 * group of G = Hq / Hkv query heads is split into, is the smallest divisor of G above 1
 * that brings the items to 256 or more, else G. A pure function of the sizes. */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                        attn_dtype_t dtype);

/* Size of the library's static device scratch array used by attn_bwd_noalloc: 8 MiB.
 * A problem fits when attn_bwd_workspace_size(...) <= ATTN_NOALLOC_SCRATCH_BYTES: delta
 * takes 4 bytes per query row (B * Hq * Sq <= 2,097,152 rows when nothing else is
 * needed), and a bf16 GQA problem whose group is split (see attn_bwd_workspace_size)
 * adds two fp32 partial buffers of B * Skv * Hkv * P * D * 4 bytes each; the GQA
 * training shape B4 Hq8 Hkv2 S2048 D128 (P = 2) needs about 33.8 MB and is refused. */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * attn_bwd_noalloc - the backward for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for integration only.
 *
 * Some callers have no way to obtain device scratch at call time: a host that has
 * reserved all device memory for its own pool and hands an operator only its input and
 * output buffers, or a latency-critical loop that must not call cudaMalloc/cudaFree
 * because those calls can synchronize the device and stall other streams. This entry
 * point takes the same arguments as attn_bwd minus the workspace and uses a scratch
 * array that lives in the library itself (a static __device__ array of
 * ATTN_NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library until the process
 * exits). It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - Size limit: when attn_bwd_workspace_size() for these sizes exceeds
 *   ATTN_NOALLOC_SCRATCH_BYTES (delta, plus the fp32 partial dK/dV of a split GQA group)
 *   it returns ATTN_ERR_WORKSPACE and launches nothing.
 * - Set-up: the first call on a device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress); make that first call before any stream
 *   capture begins.
 * - Sharing: every call on a device uses the same array, which keeps whatever the last
 *   call left in it. Each call rewrites all the scratch it reads (delta, and every row
 *   of the partial dK/dV buffers), so nothing has to start at zero. Calls whose GPU work can overlap (different streams, or threads
 *   without ordering between them) race on the array and produce wrong gradients: issue
 *   them on one stream, or order them with events.
 * Everything else (arguments, layout, results, errors) is as for attn_bwd, whose code
 * path it runs.
 */
ATTN_API attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                        const void* o, const void* dout, const float* lse,
                                        void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                        int Sq, int Skv, int D, float scale, int causal,
                                        const int32_t* kv_lens, attn_dtype_t dtype,
                                        attn_stream_t stream);

/*
 * Waits for `stream`, then reads and clears the current device's error word.
 * Writes the raw ATTN_DEVERR_* bits to *bits when bits is not NULL. Returns
 * ATTN_ERR_TIMEOUT if the timeout bit was set, else ATTN_ERR_CUDA if the layout bit was
 * set, ATTN_ERR_INVALID_ARG if only the kv_lens or page bit was set, ATTN_OK if the word
 * was clear, ATTN_ERR_CUDA on a CUDA error.
 */
ATTN_API attn_status_t attn_peek_device_error(uint32_t* bits, attn_stream_t stream);

/* The CUDA runtime's description of the last CUDA error behind an ATTN_ERR_CUDA
 * returned to the calling thread ("no CUDA error" if none); a static string. */
ATTN_API const char* attn_last_cuda_error(void);

/* A static, human-readable name of a status code. */
ATTN_API const char* attn_status_string(attn_status_t status);

/* The library's build identity (kernel families compiled in), a static string. */
ATTN_API const char* attn_build_info(void);

/*
 * Test-only fault injection: the next bf16 forward launch applies `mask` (bit 0: its
 * producer skips its first K tile load, so the consumer's bounded wait runs out) and
 * gives up a barrier wait after `timeout_ms` (0 = the default of 4 s). The kernel then
 * records ATTN_DEVERR_TIMEOUT, lets its in-flight copies and MMAs finish, frees its
 * tensor memory and returns; attn_peek_device_error() reports ATTN_ERR_TIMEOUT. Not for
 * production use: the outputs of that call are invalid.
 */
ATTN_API void attn_test_inject_fault(uint32_t mask, uint32_t timeout_ms);

/* The number of kernel launches this library has issued in this process (all devices,
 * all threads); a monotonically increasing host-side counter. */
ATTN_API uint64_t attn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
