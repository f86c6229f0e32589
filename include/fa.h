/*
 * fa.h - C ABI of the GB300 (sm_103a) exact softmax attention library.
 *
 * Computes, for every batch b and head h (Q, K, V in R^{N x d}):
 *   S = scale * Q K^T, with S_ij = -inf for j > i when causal,
 *   P = softmax(S) (row-wise), O = P V, L_i = log sum_j exp(S_ij)   (natural log)
 * and the gradients of a scalar loss given dO = dLoss/dO:
 *   D_i = sum_k dO_ik O_ik, dV = P^T dO, dP = dO V^T, dS = P o (dP - D),
 *   dQ = scale * dS K, dK = scale * dS^T Q.
 *
 * Sources (web pages on FlashAttention-2, by title and section):
 *   "FlashAttention 2: Faster Attention with Better Parallelism and Work
 *   Partitioning" (reading note, papers.chlience.com): section 1 for the
 *   standard attention definition; 5.1-5.2 for the blocked forward with the
 *   unscaled accumulator and the stored logsumexp L = m + log(l); 5.3 for the
 *   recomputation backward with D = rowsum(dO o O).
 *   "FlashAttention" (llm-infra-atlas), section 1, for the 1/sqrt(d) scale.
 *   "FlashAttention-2: ..." (paper-graph-ui summary), "Causal masking
 *   optimization": entries whose column index exceeds the row index are -inf.
 *   Reading note 5.6 for grouped / multi-query K/V heads (fa_*_gqa).
 *
 * Conventions shared by every entry point:
 *   - Tensors are contiguous, row-major [B][H][N][d]; q, k, v, o, dO, dq, dk,
 *     dv are bfloat16; lse is float32 [B][H][N]. All are DEVICE pointers
 *     owned by the caller. bf16 pointers must be 16-byte aligned, lse 4-byte
 *     aligned, the workspace 256-byte aligned.
 *   - d must be 64, 128 or 256 (else FA_ERR_UNSUPPORTED). N >= 0, B >= 0,
 *     H >= 0; if B*H*N == 0 the call does nothing and returns FA_OK (null
 *     pointers are then allowed). scale must be finite and > 0.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).
 *     Argument errors are returned synchronously before any GPU work is
 *     queued. Launch failures return FA_ERR_LAUNCH / FA_ERR_CUDA.
 *   - Device-side failures (a pipeline wait that exceeded its time limit) are
 *     recorded in a per-device status word that fa_get_device_status() reads.
 *   - The library allocates no device memory; it keeps only cached device
 *     attributes in process-wide state (plus, once fa_fwd_bwd_host or
 *     fa_fwd_host has run on a device, twelve streams and 50 events for
 *     that device; they serve one call at a time). Entry points are
 *     thread-safe.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale or flag */
  FA_ERR_UNSUPPORTED = 2, /* head dimension other than 64/128/256, or no sm_103a device */
  FA_ERR_MISALIGNED = 3,  /* pointer alignment below the stated minimum */
  FA_ERR_WORKSPACE = 4,   /* backward workspace missing or too small */
  FA_ERR_LAUNCH = 5,      /* a kernel launch failed */
  FA_ERR_TIMEOUT = 6,     /* a device-side pipeline wait gave up (see fa_get_device_status) */
  FA_ERR_CUDA = 7         /* another CUDA runtime error */
} fa_status_t;

/*
 * Forward pass (reading note 5.1-5.2; paper-graph-ui summary, "Algorithm 1
 * Walkthrough"): O = softmax(scale * Q K^T [causal]) V and L = logsumexp per
 * query row.
 *   q, k, v : in,  bf16 [B][H][N][d]
 *   o       : out, bf16 [B][H][N][d]
 *   lse     : out, fp32 [B][H][N], natural log, in units of the scaled scores
 *   causal  : 0 or 1
 *   scale   : softmax scale, typically 1/sqrt(d)
 */
fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   int causal, float scale, cudaStream_t stream);

/*
 * Forward pass with grouped / multi-query K/V heads (reading note 5.6;
 * paper-graph-ui summary, "Multi-query and grouped-query attention"): Hq query
 * heads share Hkv K/V heads, g = Hq / Hkv query heads per K/V head, and query
 * head h reads K/V head floor(h / g). Nothing is copied.
 *   q, o    : bf16 [B][Hq][N][d];  lse : fp32 [B][Hq][N]
 *   k, v    : bf16 [B][Hkv][N][d]
 *   Hkv     : >= 1 and dividing Hq (else FA_ERR_INVALID_ARG); Hkv == Hq is fa_fwd.
 * Other arguments and errors as for fa_fwd.
 */
fa_status_t fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int N, int d, int causal, float scale, cudaStream_t stream);

/*
 * Forward pass over a key range split and/or a key sequence of its own
 * length (a query block against a longer key/value cache, e.g. decoding):
 *   q, o : bf16 [B][Hq][Nq][d];  lse : fp32 [B][Hq][Nq]
 *   k, v : bf16 [B][Hkv][Nk][d]  (grouped heads as for fa_fwd_gqa)
 *   causal : query i sees key j iff j <= i + (Nk - Nq), i.e. the mask is
 *            aligned to the last key (for Nq = Nk the usual causal mask);
 *            needs Nq <= Nk. Nk must be >= 1.
 *   num_splits : the keys of each query tile are cut into this many ranges of
 *            whole 128-key tiles, processed as separate work items, and the
 *            partial results (O of each range normalised by its own sum, and
 *            its logsumexp L_s) are merged by a combine kernel:
 *              L = log sum_s e^{L_s},  O = sum_s e^{L_s - L} O_s
 *            (reading note 5.2: the running max and sum make softmax blocks
 *            combinable). 1: no split, no workspace. 0: the library chooses,
 *            within the workspace given. At most 256; ranges beyond the keys
 *            are dropped.
 *   workspace : fa_fwd_splitkv_workspace_size(B, Hq, Nq, d, splits) bytes,
 *            256-byte aligned, for any split count above 1.
 */
fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, int causal, float scale, int num_splits, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);
size_t fa_fwd_splitkv_workspace_size(int B, int Hq, int Nq, int d, int num_splits);

/*
 * Bytes of device workspace fa_bwd needs: D and the base-2 logsumexp
 * (fp32 per query row) and the fp32 dQ accumulator, with every head padded
 * to a multiple of 128 rows, plus 256 bytes for the main kernel's work-item
 * counter. Returns 0 for invalid or empty sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass (reading note 5.3; paper-graph-ui summary, "The Backward
 * Pass"): recomputes S and P = exp(S - L) block by block, then
 *   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
 *   dK = scale dS^T Q, with D = rowsum(dO o O) precomputed.
 *   q, k, v, o : in, bf16 [B][H][N][d] (o is the forward output)
 *   lse        : in, fp32 [B][H][N] from fa_fwd with the same arguments
 *   dO         : in, bf16 [B][H][N][d]
 *   dq, dk, dv : out, bf16 [B][H][N][d]
 *   workspace  : device scratch of at least fa_bwd_workspace_size() bytes,
 *                owned by the caller; its contents on entry do not matter.
 * dQ: for d = 64 and 256 it is accumulated in fp32 with atomic adds across
 * key blocks (the pages' scheme), so dq is not bitwise reproducible run to
 * run; for d = 128 fa_bwd runs the sequence of fa_bwd_deterministic, which
 * measured faster at that head dimension, and dq is reproducible. dk and dv
 * are always reproducible.
 */
fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward pass with grouped / multi-query K/V heads (reading note 5.6): the
 * gradient of a shared K/V head is the sum over its g query heads,
 *   dK_{h_kv} = sum over h with floor(h / g) = h_kv of dK_h (same for dV).
 * A work item accumulates one key tile's dK, dV on chip over a chunk of the g
 * query heads. When the problem has too few (K/V head, key tile) pairs to
 * fill the GPU, or, under a causal mask, too long an item, the library
 * splits each group into chunks; their fp32 partial sums go to the workspace
 * and a post kernel adds them in chunk order. Either way dk and dv are
 * bitwise reproducible.
 *   q, o, dO, dq : bf16 [B][Hq][N][d];  lse : fp32 [B][Hq][N]
 *   k, v, dk, dv : bf16 [B][Hkv][N][d]
 *   workspace    : at least fa_bwd_workspace_size(B, Hq, N, d) bytes; the
 *                  group is split only as far as the bytes beyond that allow
 *                  (fa_bwd_gqa_workspace_size leaves room for every split).
 * Other arguments and errors as for fa_bwd; Hkv == Hq is fa_bwd.
 */
size_t fa_bwd_gqa_workspace_size(int B, int Hq, int Hkv, int N, int d);

/*
 * Deterministic backward: the same results as fa_bwd / fa_bwd_gqa, but dq is
 * bitwise reproducible too. The pages accumulate dQ_i += dS K_j across key
 * blocks with atomic adds (reading note 5.3-5.4; paper-graph-ui summary, "The
 * Backward Pass"), whose order varies run to run. Here a separate kernel owns
 * each 128-row query tile, recomputes S, P, dP and dS for every key tile it
 * sees and sums dQ_i on chip in key order; the main kernel then computes only
 * dK and dV. Costs three more 128x128xd products per (query tile, key tile)
 * pair than the atomic version.
 *   Arguments, layouts and workspace as for fa_bwd / fa_bwd_gqa.
 *   d = 64, 128 or 256 (at d = 256 the dQ kernel streams K and V in 64-column
 *   chunks and reads K twice, since Q, dO and a 128-key K tile do not fit in
 *   shared memory together).
 */
fa_status_t fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                 const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                                 float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status_t fa_bwd_gqa_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                     const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                                     int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream);

fa_status_t fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d,
                       int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The three phases fa_bwd runs, in order, on one stream (each also callable on
 * its own with the same sizes and workspace; fa_bwd == preprocess, main,
 * postprocess). Arguments mean what they mean for fa_bwd.
 *
 * fa_bwd_preprocess: D_i = sum_k dO_ik O_ik (the row-wise correction that
 *   reading note 5.3 precomputes before the block loops), the base-2 logsumexp
 *   L_i * log2(e), a zeroed fp32 dQ accumulator and a zeroed work-item
 *   counter, all in the workspace.
 *   Reads o, lse, dO. HBM-bound.
 * fa_bwd_preprocess_stats: fa_bwd_preprocess without zeroing the dQ
 *   accumulator (D, the base-2 logsumexp and the work-item counters only):
 *   the first phase of fa_bwd_deterministic, whose dQ kernel does not use
 *   the accumulator. Same arguments.
 * fa_bwd_main: the block loops of reading note 5.3 (key blocks outer): writes
 *   dk and dv, and adds every dS K_j into the workspace's dQ accumulator.
 *   Reads q, k, v, dO and the preprocessed workspace.
 * fa_bwd_postprocess: dq = bf16(dQ accumulator). HBM-bound.
 */
fa_status_t fa_bwd_preprocess(const void* o, const float* lse, const void* dO, int B, int H, int N, int d,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status_t fa_bwd_preprocess_stats(const void* o, const float* lse, const void* dO, int B, int H, int N, int d,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status_t fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B,
                        int H, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);
/*
 * The phases of the deterministic backward (d = 64, 128, 256), run after
 * fa_bwd_preprocess_stats (or fa_bwd_preprocess) on the same workspace:
 * fa_bwd_deterministic == preprocess_stats, dkdv, dq.
 * fa_bwd_dkdv: the block loops of reading note 5.3 without the dQ products:
 *   writes dk and dv.
 * fa_bwd_dq: per 128-row query tile, recomputes S, P, dP and dS for every key
 *   tile it sees and sums dQ on chip in key order; writes dq.
 * Within fa_bwd_deterministic (and fa_bwd at d = 128) the dQ kernel is
 * launched to overlap the dK/dV kernel before it on the stream (programmatic
 * dependent launch: it takes the SMs the dK/dV pass leaves idle in its last
 * round) and completes only after that kernel has, so work queued after the
 * call sees dq, dk and dv final. The separate entry points launch without
 * the overlap; an event recorded between them would serialise it anyway.
 * The dK/dV kernel signals programmatic launch completion at its start, so a
 * kernel a caller queues after fa_bwd_dkdv with programmatic stream
 * serialization must wait for its prerequisite grid (as that launch mode
 * always requires) before it reads dk or dv; ordinary launches are ordered
 * as usual.
 */
fa_status_t fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B,
                        int H, int N, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);
fa_status_t fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B, int H, int N,
                      int d, int causal, float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);
fa_status_t fa_bwd_postprocess(void* dq, int B, int H, int N, int d, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * Backward pass for callers that cannot allocate device memory. This entry
 * point has no counterpart in the paper; it is a convenience of this library.
 *
 * Some callers are handed only their input and output buffers and have no
 * allocator of their own: plugin hooks of inference engines and runtimes that
 * plan every device byte up front and forbid allocations afterwards, or code
 * that must not call cudaMalloc because it can synchronise the device and
 * stall other work. fa_bwd needs a caller-provided workspace; this variant
 * instead uses a scratch array compiled into the library (a file-scope
 * __device__ array of FA_BWD_NOALLOC_SCRATCH_BYTES, which every GPU that
 * loads the library holds until the process exits).
 *
 *   Arguments and results are those of fa_bwd, minus the workspace.
 *   Problems whose workspace (fa_bwd_workspace_size) exceeds
 *   FA_BWD_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_WORKSPACE before
 *   any GPU work; use fa_bwd with your own workspace for those. That size
 *   always counts the fp32 dQ accumulator (4 d bytes per padded row), also at
 *   d = 128 where fa_bwd forms dQ without it, so at d = 128 the largest
 *   accepted problem is about 32k padded rows (B * H * ceil(N / 128) * 128).
 *   A device that is not sm_103a gives FA_ERR_UNSUPPORTED, as for fa_bwd.
 *   The call allocates nothing: no cudaMalloc/cudaFree and no allocating
 *   library routine.
 *   The first call on a device looks up the scratch array's device address
 *   (once per device, with that device current; a failed lookup is retried
 *   by the next call); make that first call before any stream capture.
 *   All calls share the one array per device. Each call re-initialises the
 *   parts that must start at zero, so a call never sees the previous call's
 *   values, but calls that overlap on the GPU (different streams or
 *   threads without ordering between them) race on the array and give wrong
 *   results.
 */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
fa_status_t fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                           float scale, cudaStream_t stream);

/*
 * Forward and backward pass of a problem held in HOST memory (the forward of
 * reading note 5.1-5.2 and the backward of 5.3, as fa_fwd and fa_bwd), with
 * the host<->device copies overlapped with the kernels.
 *   q, k, v, dO     : in,  HOST bf16 [B][H][N][d]
 *   o               : out, HOST bf16 [B][H][N][d]
 *   lse             : out, HOST fp32 [B][H][N]
 *   dq, dk, dv      : out, HOST bf16 [B][H][N][d]
 *   device_buffer   : DEVICE memory of at least
 *                     fa_fwd_bwd_host_device_bytes(B, H, N, d) bytes,
 *                     256-byte aligned, owned by the caller; it receives the
 *                     device copies and the backward workspace, and its
 *                     contents are undefined afterwards.
 * Host buffers may have any alignment. The copies overlap the kernels only
 * when the host buffers are page-locked (cudaHostAlloc / cudaHostRegister);
 * pageable buffers give the same results with serialised copies.
 * The call splits the B*H heads into up to four groups (by default an eighth
 * of the heads, two groups holding the rest halved, and another eighth) and
 * queues, in order after the work already on `stream`: the uploads of each
 * group's Q, K, V (the middle groups' in two chunks of heads) and dO on a
 * library-owned copy stream; the forward per chunk as soon as its inputs are
 * on the device, on two library-owned streams at the greatest priority; per
 * group, on its own library-owned streams and its own part of device_buffer,
 * the backward phases fa_bwd runs for this d (d = 128: the dK/dV and dQ
 * kernels side by side); the read-back of O and L, dK and dV, and dQ of each
 * group as soon as each is final, on a second copy stream. Later groups'
 * uploads thus overlap earlier groups' kernels, and one launch's last,
 * partly empty round fills with another's work. Work queued on `stream`
 * after the call, and a synchronisation of `stream`, see every output in
 * host memory. Only equal-head problems (one K/V head per query head).
 * Errors: those of fa_fwd / fa_bwd, checked before any work is queued;
 * FA_ERR_WORKSPACE if device_buffer is null or too small, FA_ERR_MISALIGNED
 * if it is not 256-byte aligned, FA_ERR_CUDA if a copy or an event call
 * fails (the outputs are then undefined).
 */
size_t fa_fwd_bwd_host_device_bytes(int B, int H, int N, int d); /* 0 for invalid or empty problems */
fa_status_t fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                            void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                            void* device_buffer, size_t device_bytes, cudaStream_t stream);

/*
 * Forward pass of a problem held in HOST memory (as fa_fwd), pipelined over
 * eight chunks of heads: while chunk c is on the tensor cores, chunk c + 1
 * uploads and chunk c - 1 is read back. The chunks' launches alternate
 * between two library-owned streams, so one fills the last round of the
 * one before.
 *   q, k, v         : in,  HOST bf16 [B][H][N][d]
 *   o               : out, HOST bf16 [B][H][N][d]
 *   lse             : out, HOST fp32 [B][H][N]
 *   device_buffer   : DEVICE memory of at least
 *                     fa_fwd_host_device_bytes(B, H, N, d) bytes, 256-byte
 *                     aligned, owned by the caller (undefined afterwards).
 * Host buffers, streams, ordering and errors as for fa_fwd_bwd_host.
 */
size_t fa_fwd_host_device_bytes(int B, int H, int N, int d); /* 0 for invalid or empty problems */
fa_status_t fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                        int causal, float scale, void* device_buffer, size_t device_bytes, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status_t status);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * Returns FA_OK, FA_ERR_TIMEOUT if a kernel's bounded wait gave up since the
 * last call, or FA_ERR_CUDA if the synchronisation failed.
 */
fa_status_t fa_get_device_status(cudaStream_t stream);

/*
 * As fa_get_device_status, and also copies the whole status word into
 * word[4] (host memory, owned by the caller): word[0] the status code,
 * word[1] the role of the thread whose wait gave up first (1-3: forward
 * load / MMA / softmax; 11-14: backward load / MMA / softmax / dQ drain;
 * 99: the self-test probe), word[2] its block index, word[3] its thread
 * index; all zero when no wait gave up. Returns FA_ERR_INVALID_ARG for a
 * null word.
 */
fa_status_t fa_get_device_status_detail(unsigned int* word, cudaStream_t stream);

/*
 * Time limit, in nanoseconds, of every device-side pipeline wait in later
 * launches (default 4e9; 0 restores the default; values above 1e10 are
 * capped at 1e10, so a stalled pipeline always gives up within 10 s). A wait
 * that exceeds it records FA_ERR_TIMEOUT and the kernel returns early with
 * its outputs undefined.
 */
void fa_set_wait_limit_ns(unsigned long long limit_ns);

/*
 * Failure-detection self-test: launches one CTA that waits on a barrier no
 * thread ever arrives at, with the given limit, so the wait gives up and
 * records FA_ERR_TIMEOUT. Asynchronous; read the result with
 * fa_get_device_status().
 */
fa_status_t fa_debug_timeout_probe(unsigned long long limit_ns, cudaStream_t stream);

/*
 * Failure-detection test hook for the real kernels. Off (0) by default. With
 * a role code of fa_get_device_status_detail (1-3 forward load / MMA /
 * softmax; 11-14 backward load / MMA / softmax / dQ drain), block 0 of every
 * later launch of a kernel that has that role misses one of that role's
 * hand-offs: a load role leaves out one of its TMA copies; for an MMA,
 * softmax or dQ-drain role, one barrier it signals is set up to expect one
 * arrival more than the role makes. Either way the bounded wait on that
 * barrier gives up after the wait limit: the launch records
 * FA_ERR_TIMEOUT, lets every copy and MMA it issued complete, frees its
 * tensor memory and returns, and its outputs are undefined. Other blocks run
 * normally. fa_debug_skip_arrival(0) turns the hook off. Process-wide; meant
 * for tests (set a short limit with fa_set_wait_limit_ns first).
 * FA_ERR_INVALID_ARG for any other value.
 */
fa_status_t fa_debug_skip_arrival(unsigned int role);

/* Library version, major*10000 + minor*100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
