/*
 * libsdpa: fused scaled dot-product attention and multi-head attention on
 * one GB300 GPU (sm_103a), behind a plain C ABI.
 *
 * The operations are those of "Attention Is All You Need":
 *   section 3.2.1, Eq. (1):  Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   section 3.2.3:           illegal (future) connections of the decoder's
 *                            self-attention are set to -infinity before the
 *                            softmax, so position i sees keys j <= i
 *   section 3.2.2:           MultiHead(Q, K, V) = Concat(head_1..head_h) W^O,
 *                            head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V)
 *
 * Conventions shared by every entry point:
 *   - Pointers named as device pointers are CUDA device addresses on the
 *     current device, owned by the caller; the library keeps no reference
 *     after the call returns and allocates no memory on the call path.
 *   - Tensors are dense and row-major; every device pointer must be 16-byte
 *     aligned (the kernels move tiles with the Tensor Memory Accelerator).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  A successful return means the work was
 *     enqueued; errors detected on the host are returned before anything is
 *     enqueued.  The attention, projection, backward-convert and decode-
 *     combine kernels launch with a programmatic dependency on the kernel
 *     before them in the stream: they may start setting up while it
 *     finishes, but read or write no global memory until it has completed,
 *     so stream order is kept.
 *   - Masks (`mask_kind`, bit flags): SDPA_MASK_CAUSAL hides keys j > i (it
 *     requires n_q == n_k); SDPA_MASK_PADDING hides keys j >= kv_lengths[b]
 *     (`kv_lengths`: device int32 [b], values clamped into [0, n_k] on the
 *     device).  A query row with no visible key returns a row of zeros.
 *   - `scale` multiplies Q K^T; 0.0f selects 1/sqrt(d_k) (Eq. (1)); 1.0f gives
 *     the unscaled dot-product attention of section 3.2.1.  It must be >= 0
 *     and finite.
 *   - Per-device state (the device check, the address of the kernels' error
 *     word, the static array of mha_forward_noalloc) is set up by the first
 *     call on each device and cached.  It belongs to the device's primary
 *     context: after cudaDeviceReset, or anything else that destroys that
 *     context, the process must not call the library again.
 */
#ifndef LIBSDPA_SDPA_H
#define LIBSDPA_SDPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, misalignment, bad mask */
  SDPA_ERR_UNSUPPORTED = 2,        /* valid but outside what the kernels implement */
  SDPA_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or not an sm_103 GPU */
  SDPA_ERR_WORKSPACE = 4,          /* workspace null or smaller than mha_workspace_size() */
  SDPA_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
  SDPA_ERR_DEVICE_TIMEOUT = 6      /* a kernel gave up on a bounded wait (sdpa_device_check) */
} sdpa_status;

enum { SDPA_MASK_NONE = 0, SDPA_MASK_CAUSAL = 1, SDPA_MASK_PADDING = 2 };

/*
 * Kernel choice.  The library picks each launch's kernel and tile sizes from
 * the shapes; the results agree to bf16 rounding whichever is picked, and the
 * library reads no environment variable.  For tests and tuning, this call
 * pins a choice for every later call in the process (all threads, all
 * devices) until it is called again; 0 leaves that choice to the shapes:
 *   attention_kernel  forward attention kernel for d_k == d_v <= 128:
 *       1 = one 128-row query tile per CTA, 2 = two.  By shape: one tile
 *       while a query tile sees at most 3072 keys (4352 with a restricted
 *       window), two beyond.
 *   one_tile_keys  32 | 64: key tile of the one-tile kernel at d = 64.  By
 *       shape: 32 for walks of at most 2048 keys when the grid has at least
 *       four CTAs per SM, 64 otherwise.
 *   gemm_bn  256 | 128: column tile of the projection GEMMs.  By shape: 256,
 *       or 128 when 256-column tiles would not reach half the SMs.
 * Returns SDPA_ERR_INVALID_ARG (and changes nothing) for any other value.
 * Launches already enqueued are not affected.
 */
sdpa_status sdpa_set_kernel_choice(int attention_kernel, int one_tile_keys, int gemm_bn);

/*
 * Scaled dot-product attention, bf16 (Eq. (1) with the masks above).
 *   q   [b, h, n_q, d_k]  bf16, device
 *   k   [b, h, n_k, d_k]  bf16, device
 *   v   [b, h, n_k, d_v]  bf16, device
 *   out [b, h, n_q, d_v]  bf16, device, written (must not overlap the inputs)
 * Scores, softmax statistics and the P.V accumulation are fp32; the
 * softmax weights enter P.V rounded to bf16.  Supported (else
 * SDPA_ERR_UNSUPPORTED), the head shapes of the paper's Table 3:
 *   d_k == d_v in {16, 32, 64, 128, 256, 512} (rows (A), (C));
 *   d_k in {16, 32} with d_v == 64 (rows (B): smaller keys than values).
 * 256 and 512 run on a kernel with one query tile per CTA; for 512 two CTAs
 * split d_v and both compute the scores.
 * b, h >= 1; n_q, n_k >= 0 (zero-sized work returns SDPA_OK with nothing
 * enqueued; n_k == 0 writes zeros).
 */
sdpa_status sdpa_forward(const void* q, const void* k, const void* v, void* out,
                         int b, int h, int n_q, int n_k, int d_k, int d_v,
                         int mask_kind, const int32_t* kv_lengths, float scale,
                         void* stream);

/*
 * Restricted self-attention ("Attention Is All You Need", section 4): each
 * output position i considers only a neighbourhood of size r of the input
 * centred on it, read as the keys i - floor((r-1)/2) .. i + floor(r/2)
 * (exactly r positions; symmetric for odd r).  Tensors, types, masks and
 * rules as sdpa_forward; the window combines with SDPA_MASK_CAUSAL (which
 * then leaves keys i - floor((r-1)/2) .. i) and SDPA_MASK_PADDING.  Key tiles
 * outside every query's window are neither loaded nor multiplied, so the
 * cost grows as n * r instead of n^2.  r >= 1 (else SDPA_ERR_INVALID_ARG).
 */
sdpa_status sdpa_forward_restricted(const void* q, const void* k, const void* v, void* out,
                                    int b, int h, int n_q, int n_k, int d_k, int d_v,
                                    int mask_kind, const int32_t* kv_lengths, int r, float scale,
                                    void* stream);

/*
 * sdpa_forward that also returns, for the backward pass, each query row's
 * natural log-sum-exp of its scaled, masked scores:
 *   lse [b, h, n_q] fp32, device, written: lse_i = ln sum_{j visible} exp(scale q_i . k_j)
 *   (-INFINITY for a row with no visible key).
 * r = 0 is plain attention; r >= 1 is the restricted window of
 * sdpa_forward_restricted.  Otherwise as sdpa_forward (lse 4-byte aligned).
 */
sdpa_status sdpa_forward_lse(const void* q, const void* k, const void* v, void* out, float* lse,
                             int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                             const int32_t* kv_lengths, int r, float scale, void* stream);

/*
 * Gradients of scaled dot-product attention, for training the model by
 * back-propagation ("Attention Is All You Need", section 5, through Eq. (1)).
 * With S = scale Q K^T (masked entries -inf), P = softmax(S) row-wise,
 * O = P V and the upstream gradient dO:
 *   dV = P^T dO,   dP = dO V^T,   dS = P o (dP - rowsum(dO o O)),
 *   dQ = scale dS K,   dK = scale dS^T Q.
 *   q, k, v, out  the forward's bf16 BHSD inputs and output, device
 *   dout [b, h, n_q, d_v] bf16, device: the gradient of the loss w.r.t. out
 *   lse  [b, h, n_q] fp32, device: sdpa_forward_lse's output for this call
 *   dq [b, h, n_q, d_k], dk [b, h, n_k, d_k], dv [b, h, n_k, d_v] bf16,
 *        device, written (must not overlap the inputs or one another)
 *   workspace: device buffer of ws_bytes >= sdpa_backward_workspace_size(b, h,
 *        n_q, d_k), 16-byte aligned, caller-owned (fp32 dQ accumulator and
 *        per-row vectors); reusable once the stream passes the call.
 *   mask_kind, kv_lengths, r, scale: the values given to the forward.
 * P is recomputed from lse, never stored; the products run on the tensor
 * cores with bf16 operands (P and dS rounded to bf16) and fp32 accumulation;
 * dQ is accumulated in fp32 across key tiles, then rounded.  Hidden keys get
 * zero gradient.  Supported: d_k == d_v in {16, 32, 64, 128, 256, 512}
 * (every head size of Table 3), and (d_k, d_v) in {(16, 64), (32, 64)}
 * (Table 3, rows (B)); other sizes return SDPA_ERR_UNSUPPORTED.
 * The forward output `out` enters only through D_i = dO_i . out_i.
 */
size_t sdpa_backward_workspace_size(int b, int h, int n_q, int d);

sdpa_status sdpa_backward(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          void* workspace, size_t ws_bytes, int b, int h, int n_q, int n_k,
                          int d_k, int d_v, int mask_kind, const int32_t* kv_lengths, int r,
                          float scale, void* stream);

/*
 * The bf16 attention of sdpa_forward over HOST buffers, for callers whose
 * inputs and outputs live in host memory (section 3.2.1, Eq. (1), with the
 * masks above).
 *   q_host, k_host, v_host, out_host: BHSD bf16 host buffers, shapes as in
 *     sdpa_forward; page-locked (cudaHostAlloc / cudaHostRegister) for the
 *     copies to run asynchronously and overlap; pageable memory works but
 *     each copy then blocks the calling thread.
 *   q_dev, k_dev, v_dev, out_dev: caller-owned device buffers of the same
 *     shapes, used as staging; they hold the inputs and the output after
 *     the call completes.
 *   heads_per_chunk: the work is cut into (batch entry, heads_per_chunk
 *     heads) chunks (0: all heads of a batch entry).  Each chunk's copy in,
 *     attention and copy out go on three streams of the library's own, so
 *     the copies of one chunk overlap the attention of another.
 *   stream: the work starts after what is queued on `stream`, and `stream`
 *     waits for the last copy back: synchronise it before reading out_host.
 * The first call on a device creates the library's three streams and four
 * events there, kept for the process; concurrent calls on one device are
 * serialised on the host while they enqueue.  Argument rules and statuses
 * are sdpa_forward's, plus SDPA_ERR_INVALID_ARG for a null host pointer or a
 * negative heads_per_chunk; they are checked before anything is enqueued.
 * If a CUDA call fails while the chunks are being enqueued, the call returns
 * SDPA_ERR_CUDA at once: chunks enqueued before it may still be running on
 * the library's streams, and `stream` does not wait for them (synchronise
 * the device before reusing the buffers).
 */
sdpa_status sdpa_forward_host(const void* q_host, const void* k_host, const void* v_host,
                              void* out_host, void* q_dev, void* k_dev, void* v_dev,
                              void* out_dev, int b, int h, int n_q, int n_k, int d_k, int d_v,
                              int mask_kind, const int32_t* kv_lengths, float scale,
                              int heads_per_chunk, void* stream);

/*
 * The same operation in fp32 throughout (fp32 inputs, exact fp32 exponentials
 * and sums on the CUDA cores), for small fp32 problems and the worked
 * examples.  Layouts as sdpa_forward with float elements; any
 * 1 <= d_k, d_v <= 128.
 */
sdpa_status sdpa_forward_f32(const void* q, const void* k, const void* v, void* out,
                             int b, int h, int n_q, int n_k, int d_k, int d_v,
                             int mask_kind, const int32_t* kv_lengths, float scale,
                             void* stream);

/*
 * One autoregressive decoding step ("Attention Is All You Need", section 3.1:
 * the decoder generates one symbol at a time): 1 <= n_q <= 8 new queries per
 * (batch, head) against cached keys and values.
 *   q   [b, h, n_q, d_k]  bf16, device (the new queries)
 *   k   [b, h, n_k, d_k]  bf16, device (key cache, capacity n_k)
 *   v   [b, h, n_k, d_v]  bf16, device (value cache)
 *   out [b, h, n_q, d_v]  bf16, device, written
 *   kv_lengths: device int32 [b], the filled length len_b of each cache
 *   (clamped into [0, n_k]), or NULL for n_k.  The new queries are the last
 *   n_q positions of each sequence, so query i sees keys j <= len_b - n_q + i
 *   (the causal rule of section 3.2.3); a query with no visible key gives 0.
 *   workspace: device buffer of ws_bytes >= sdpa_decode_workspace_size(...)
 *   (may be NULL when that size is 0), 16-byte aligned, caller-owned.  The
 *   size depends on the current device's SM count: ask on the device the
 *   step runs on.
 * The step is bound by reading the caches once from HBM; it runs on the CUDA
 * cores with the cache split across CTAs and a merge of the partial softmax
 * states.  Supported (else SDPA_ERR_UNSUPPORTED), the head shapes of the
 * paper's Table 3: d_k == d_v in {16, 32, 64, 128, 256, 512}, and d_k in
 * {16, 32} with d_v = 64 (rows (B)); b * h <= 65535.
 */
size_t sdpa_decode_workspace_size(int b, int h, int n_q, int n_k, int d_v);

sdpa_status sdpa_decode(const void* q, const void* k, const void* v, void* out, void* workspace,
                        size_t ws_bytes, int b, int h, int n_q, int n_k, int d_k, int d_v,
                        const int32_t* kv_lengths, float scale, void* stream);

/*
 * Bytes of device workspace mha_forward needs: the projected Q [b*n_q, h*d_k],
 * K [b*n_k, h*d_k], V [b*n_k, h*d_v] and the concatenated heads
 * [b*n_q, h*d_v], bf16, each rounded up to 256 bytes.  Returns 0 for
 * negative sizes.
 */
size_t mha_workspace_size(int b, int n_q, int n_k, int h, int d_k, int d_v);

/*
 * Multi-head attention (section 3.2.2) without biases:
 *   Q = X_q W^Q, K = X_kv W^K, V = X_kv W^V, head i = columns [i*d, (i+1)*d),
 *   Y = Concat(head_1..head_h) W^O.
 *   xq  [b, n_q, d_model]   bf16, device (decoder queries, or the sequence)
 *   xkv [b, n_k, d_model]   bf16, device (encoder output for cross-attention;
 *                           pass xkv == xq and n_k == n_q for self-attention)
 *   wq, wk [d_model, h*d_k]; wv [d_model, h*d_v]; wo [h*d_v, d_model]  bf16, device
 *   y   [b, n_q, d_model]   bf16, device, written
 *   workspace: device buffer of ws_bytes >= mha_workspace_size(...), 16-byte
 *   aligned, owned by the caller and reusable once the stream passes the call.
 * Projections run on the tensor cores with fp32 accumulation and bf16
 * outputs; the heads are written straight into the Concat layout.
 * Supported: the (d_k, d_v) pairs of sdpa_forward; d_model a multiple of 8.
 */
sdpa_status mha_forward(const void* xq, const void* xkv, const void* wq, const void* wk,
                        const void* wv, const void* wo, void* y, void* workspace,
                        size_t ws_bytes, int b, int n_q, int n_k, int d_model, int h,
                        int d_k, int d_v, int mask_kind, const int32_t* kv_lengths,
                        float scale, void* stream);

/*
 * mha_forward for callers that cannot allocate device memory.  The paper has
 * no counterpart: this entry point exists for integration, not for the method.
 *
 * Some callers cannot call cudaMalloc, for example code inside a host
 * framework that owns all device memory through its own pool, or code on a
 * latency-critical path that must not risk the device-wide synchronisation an
 * allocation can cause.  This variant takes no workspace: it uses a static
 * device array of SDPA_MHA_NOALLOC_MAX_WORKSPACE bytes inside the library,
 * which every GPU that loads the library holds until the process exits.  The
 * caller still passes (and owns) the inputs and the output, with the same
 * meaning, layouts and rules as mha_forward.
 *   - Returns SDPA_ERR_WORKSPACE, before enqueuing anything, when
 *     mha_workspace_size(b, n_q, n_k, h, d_k, d_v) exceeds
 *     SDPA_MHA_NOALLOC_MAX_WORKSPACE.  The argument checks of mha_forward
 *     come first, so an invalid or unsupported argument returns the same
 *     status as there.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - The first call on each device looks up the array's device address and
 *     caches it; make that first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Calls that overlap on the GPU (e.g. on two streams, or from two host
 *     threads) race on it: order them on one stream or synchronise.
 */
#define SDPA_MHA_NOALLOC_MAX_WORKSPACE (32u << 20) /* bytes: 32 MiB */

sdpa_status mha_forward_noalloc(const void* xq, const void* xkv, const void* wq, const void* wk,
                                const void* wv, const void* wo, void* y, int b, int n_q, int n_k,
                                int d_model, int h, int d_k, int d_v, int mask_kind,
                                const int32_t* kv_lengths, float scale, void* stream);

/*
 * One projection of section 3.2.2 on its own: y[m, n] = sum_k x[m, k] w[k, n],
 * x [m, k], w [k, n], y [m, n] bf16 row-major device tensors, fp32
 * accumulation.  k and n must be multiples of 8; m, n, k >= 1.
 */
sdpa_status linear_forward(const void* x, const void* w, void* y, int m, int n, int k,
                           void* stream);

/*
 * Waits for the current device to finish its queued work, then reads and
 * clears the kernels' error word.  Returns SDPA_ERR_DEVICE_TIMEOUT if a
 * kernel abandoned a bounded wait since the last check (its output is then
 * undefined), SDPA_ERR_CUDA if the synchronisation failed, else SDPA_OK.
 */
sdpa_status sdpa_device_check(void);

/* A static, human-readable name for a status code. */
const char* sdpa_status_string(sdpa_status status);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* LIBSDPA_SDPA_H */
