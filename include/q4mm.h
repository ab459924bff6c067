/*
 * q4mm — GB300 (sm_103a) kernels for the Linear-layer product y = x·Wᵀ with
 * an FP32 activation and a block-quantized weight that is dequantized inside
 * the kernel.  C ABI of libq4mm.so.
 *
 * Shapes and layouts (every entry point):
 *   K = inputDim, N = outputDim, T = tokens.
 *   x  : T rows of K fp32 values, row-major ([T][K]); token r starts at x + r·K.
 *   W  : N output rows stored one after another ([out, in] order, used in
 *        place, never transposed; SKaiNET docs "Eager execution: backends and
 *        kernels", paragraph on the dense x·Wᵀ row).  Each row is a run of
 *        contiguous blocks (the BLOCKED_ROW_MAJOR order of SKaiNET issue
 *        #1138, section "Tasks").
 *   y  : T rows of N fp32 values, row-major ([T][N]); token r writes y + r·N
 *        (the prefill loop "advance offsets by r·k / r·n", same section).
 *        y is overwritten, never accumulated into.
 *
 * Ownership and memory: x, W and y are DEVICE pointers owned by the caller
 * and must not overlap.  q4k_matmul and ternary_gemv allocate nothing;
 * q4k_matmul_tc takes stream-ordered scratch for the length of each call
 * above 128 tokens (its entry below gives the size).
 *
 * Streams: every compute call is asynchronous on `stream` (NULL means the
 * legacy default stream).  Validation is synchronous: an invalid call returns
 * its error before anything is launched and leaves y untouched.  Calls on one
 * stream may overlap their prologue with the previous kernel on that stream
 * (programmatic dependent launch): weight bytes, which no earlier kernel
 * writes, may be fetched before the previous kernel has finished; x is read
 * and y written only after it has.
 *
 * Errors: every entry point returns Q4MM_OK (0) or a negative q4mm_status;
 * q4mm_last_error() then returns a message for the calling thread.  No C++
 * exception crosses this boundary.  Asynchronous faults surface through the
 * CUDA runtime as usual (the next synchronising call on the stream).
 */
#ifndef Q4MM_H
#define Q4MM_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *q4mm_stream_t;

typedef enum {
    Q4MM_OK = 0,
    Q4MM_ERR_DIM = -1,     /* a dimension is <= 0, above its limit, or inputDim breaks its multiple */
    Q4MM_ERR_NULL = -2,    /* a required pointer is NULL */
    Q4MM_ERR_ALIGN = -3,   /* a pointer is not aligned as its entry point requires */
    Q4MM_ERR_CUDA = -4,    /* the CUDA runtime reported an error (launch, device query) */
    Q4MM_ERR_TIMEOUT = -5, /* a bounded in-kernel wait ran out (see q4mm_device_status) */
    Q4MM_ERR_ALIAS = -6    /* x, W and y overlap */
} q4mm_status;

/* Largest inputDim accepted by every entry point. */
#define Q4MM_MAX_INPUT_DIM 65536

/*
 * q4k_matmul — y = x·Wᵀ with W in Q4_K, FP32 arithmetic.
 *
 * Defined by SKaiNET PR #562 "feat(kernel): SIMD-fused Q4_K matmul kernel +
 * Q4KMatmulKernel SPI": section "Pipeline" (the 256-value super-block, the
 * strided nibble layout with sub-block 2j in the low nibbles and 2j+1 in the
 * high nibbles of the same 32 bytes, value = d·sc·q − dmin·m, and the lazy
 * correction acc += scale·codeSum − offset·inputSum) and section "Test plan"
 * (inputDim must be a multiple of 256; results within 1e-4 relative of the
 * dequantize-then-matmul reference).
 *
 * w_q4k : N·(K/256) blocks of 144 bytes: fp16 d (little-endian), fp16 dmin,
 *         12 bytes packing eight 6-bit scales and eight 6-bit mins (ggml
 *         canonical packing), 128 bytes of 4-bit codes.  16-byte aligned.
 * x     : 16-byte aligned.  y: 4-byte aligned.
 * Limits: inputDim a positive multiple of 256 and <= Q4MM_MAX_INPUT_DIM;
 *         outputDim >= 1; tokens >= 1.
 * Precision: per token row t, max_o |y − y_exact| <= 1e-4 · max_o |y_exact|
 *         on the pages' test inputs and on rows with a wide dynamic range
 *         (activations of 1e5 next to ones of order 1, including on weights
 *         that are zero).  The bound behind it, up to 2 tokens: each 32-value
 *         group g of x is rounded once to a multiple of s_g·2^-23, s_g the
 *         power of two just above max_g|x|/255, i.e. to within
 *         max(2^-23·max_g|x|/255, 2^-127) (about 4.7e-10 of the group's
 *         largest magnitude; values within a factor 255 of it are exact),
 *         split into four byte planes, and the code-dots are exact integer
 *         sums; so |y_o − y_exact,o| <= Σ_g 2^-23·max_g|x|/255·Σ_{k∈g}|w_ok|
 *         plus fp32 rounding of the scales, mins and sums (relative 2^-22 or
 *         so of each term).  A large activation changes only its own group's
 *         grid.  Where that kernel's geometry does not fit (2 tokens with a
 *         large inputDim), and from 3 tokens on: fp32 dequantization and fp32
 *         fused multiply-add.
 * Weights are streamed from HBM once per call for up to 8 tokens; above
 * that once per 8 tokens (up to 32 tokens, or whenever outputDim is below
 * about 6,500 rows) or once per 64 tokens (the FP32 tile kernel).
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4k_matmul(const float *x, const void *w_q4k, float *y, int inputDim, int outputDim,
               int tokens, q4mm_stream_t stream);

/*
 * q4k_matmul_tc — the same product on the tensor cores (tcgen05), for
 * prefill-sized token counts.  The dequantized weight (computed in fp32 and
 * rounded once) and the activation are rounded to bfloat16 before the
 * multiply; products are accumulated in FP32 (tensor memory).  Same layouts,
 * alignment and limits as q4k_matmul.
 * Precision: per token row, max_o |y − y_bf16| <= 1e-4 · max_o |y_bf16| where
 * y_bf16 is the exact product of the bf16-rounded operands; the deviation
 * from the exact product is that of bf16 operand rounding (about 5e-3 of
 * max_o |y_exact| on random data).
 * Memory: up to 128 tokens a call allocates nothing (the kernel rounds x to
 * bf16 as it loads it).  Above 128 tokens each call takes stream-ordered
 * scratch (cudaMallocAsync on `stream`, released by cudaFreeAsync on
 * `stream` after the call's last kernel): the bf16 copy of x,
 * 2·tokens·inputDim bytes rounded up to 256, and the weights are read once
 * per 128 tokens.  The S = max(3, ceil(inputDim/16384)) CTAs of a cluster
 * that split the input dimension of each 256-row tile add their partial
 * sums in shared memory.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA} (CUDA also when the
 * scratch allocation fails).  A bounded wait that runs out sets the device
 * status word (see q4mm_device_status).
 */
int q4k_matmul_tc(const float *x, const void *w_q4k, float *y, int inputDim, int outputDim,
                  int tokens, q4mm_stream_t stream);

/* Largest inputDim accepted by q4_0_gemv. */
#define Q4MM_Q4_0_MAX_INPUT_DIM 32768

/*
 * q4_0_gemv — y = x·Wᵀ with W in Q4_0, FP32 result.
 *
 * The block is the one SKaiNET PR #562 names as its follow-up (section "Out
 * of scope": Q4_0, "same algorithm, simpler block", 32 values in 18 bytes).
 * The page gives no byte layout; this library reads it as ggml's: fp16 d
 * (little-endian), then 16 bytes qs; element l (l < 16) of a block is the low
 * nibble of qs[l] and element 16 + l its high nibble (the same strided
 * pattern as the Q4_K slabs); w = d·(q − 8), i.e. scale d and offset 8·d in
 * the page's lazy form.
 *
 * w_q4_0 : N·(K/32) blocks of 18 bytes, each row contiguous.  16-byte aligned.
 * x      : 16-byte aligned.  y: 4-byte aligned.
 * Limits: inputDim a positive multiple of 256 and <= Q4MM_Q4_0_MAX_INPUT_DIM
 *         (the one-token kernel's geometry: 256 values occupy 144 bytes of a
 *         row, as in Q4_K); outputDim >= 1; tokens >= 1.
 * Precision: as the one-token path of q4k_matmul: per token row,
 *         max_o |y − y_exact| <= 1e-4 · max_o |y_exact|, with x rounded once
 *         to within 2^-23/255 of each 32-value group's largest magnitude and
 *         the code-dots exact integer sums of (q − 8)·x̂, so a zero weight
 *         (q = 8) adds nothing whatever its activation.
 * Tokens: up to 8 tokens share one pass over the weights (more tokens
 *         take one pass per 8).
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4_0_gemv(const float *x, const void *w_q4_0, float *y, int inputDim, int outputDim,
              int tokens, q4mm_stream_t stream);

/* Largest inputDim accepted by q6k_gemv. */
#define Q4MM_Q6K_MAX_INPUT_DIM 32768

/*
 * q6k_gemv — y = x·Wᵀ with W in Q6_K, FP32 result.
 *
 * The block is the second follow-up SKaiNET PR #562 names (section "Out of
 * scope": Q6_K, "ql + qh with the 4-codes-per-qh-byte half-interleaved
 * layout").  The page gives no byte layout; this library reads it as ggml's:
 * 256 values in 210 bytes — ql[128] (low 4 bits of each 6-bit code), qh[64]
 * (high 2 bits, four codes per byte), 16 signed 8-bit sub-block scales, fp16
 * d (little-endian) last.  In half n (values 128n..128n+127), value
 * 128n + 32g + l (g = 0..3, l < 32) takes the low nibble of ql[64n + l]
 * (g = 0) or of ql[64n + 32 + l] (g = 1), the high nibble of ql[64n + l]
 * (g = 2) or of ql[64n + 32 + l] (g = 3), and bits 2g..2g+1 of qh[32n + l];
 * its sub-block is 8n + 2g + l/16 and w = d·scale·(q − 32).
 *
 * w_q6k : N·(K/256) blocks of 210 bytes, each row contiguous (rows need not
 *         start on a 16-byte boundary).  The buffer is 16-byte aligned.
 * x     : 16-byte aligned.  y: 4-byte aligned.
 * Limits: inputDim a positive multiple of 256 and <= Q4MM_Q6K_MAX_INPUT_DIM;
 *         outputDim >= 1; tokens >= 1 (up to 8 tokens per pass over the
 *         weights).
 * Precision: as the one-token path of q4k_matmul: per token row,
 *         max_o |y − y_exact| <= 1e-4 · max_o |y_exact|; the code-dots are
 *         exact integer sums of (q − 32)·x̂, so a zero weight adds nothing.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q6k_gemv(const float *x, const void *w_q6k, float *y, int inputDim, int outputDim, int tokens,
             q4mm_stream_t stream);

/* Largest inputDim accepted by q4k_ffn_swiglu. */
#define Q4MM_FFN_MAX_INPUT_DIM 32768

/*
 * q4k_ffn_swiglu — the input side of a Llama feed-forward block in one call:
 *   h = silu(x·W_gateᵀ) ⊙ (x·W_upᵀ),  silu(z) = z / (1 + e^(−z)),
 * both weights Q4_K (layout, values and precision as q4k_matmul's: the
 * byte-plane path for 1-2 tokens, fp32 FMA from 3 tokens on).  The pages
 * name this fused operation only as the llama.cpp benchmark "ffn_swiglu"
 * (PR #37 "ggml-cpu: cache-aware tiling in ggml_compute_forward_mul_mat",
 * section "Measured impact"); the formula is the standard Llama FFN.  For
 * 1-2 tokens one launch per token, from 3 tokens on one launch per 8 tokens,
 * each reading x once for both weights and writing only h.
 *
 * w_gate, w_up : hiddenDim rows of inputDim/256 Q4_K blocks each, 16-byte
 *                aligned; they may be the same buffer.  x: 16-byte aligned.
 *                h: [tokens][hiddenDim], 4-byte aligned, overwritten; h must
 *                not overlap x or either weight.
 * Limits: inputDim a positive multiple of 256 and <= Q4MM_FFN_MAX_INPUT_DIM;
 *         hiddenDim >= 1; tokens >= 1 (one pass over both weights per token
 *         up to 2 tokens, per 8 tokens above).
 * Precision: g and u each within q4k_matmul's bound; h = silu(g)·u
 *         in fp32 (expf), so max_o |h − h_exact| <= 1e-4 · max_o |u| ·
 *         (1.1 · max_o |g| + max_o |silu(g)|) per token (1.1 bounds |silu'|).
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4k_ffn_swiglu(const float *x, const void *w_gate, const void *w_up, float *h, int inputDim,
                   int hiddenDim, int tokens, q4mm_stream_t stream);

/* Size of the fixed device array that q4k_matmul_tc_noalloc uses as scratch. */
#define Q4MM_TC_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * q4k_matmul_tc_noalloc — q4k_matmul_tc with no allocation at all.  The pages
 * that define the product have no counterpart of this entry point.  It is for
 * callers that cannot allocate device memory while a call runs: a host
 * framework whose own allocator owns the whole device budget and forbids
 * allocations behind its back, a process on a device or driver set-up
 * without stream-ordered memory pools (where cudaMallocAsync fails), or a
 * serving loop with a latency budget that keeps allocator calls off its hot
 * path.
 *
 * Same arguments, layouts, alignment, limits, precision and results as
 * q4k_matmul_tc: the same kernels run.  The scratch that q4k_matmul_tc takes
 * per call lives instead in one fixed array of Q4MM_TC_NOALLOC_SCRATCH_BYTES
 * (16 MiB) of device memory inside the library, which every GPU that loads
 * the library holds until the process exits.  A call whose scratch (the size
 * formula under q4k_matmul_tc) is larger returns Q4MM_ERR_DIM before
 * launching anything; calls of up to 128 tokens need none, 256 tokens of a
 * 4096 → 11008 layer need 2 MiB, and the array holds up to 2048 tokens at
 * inputDim 4096.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  No part of it has to start at zero: a call writes every
 * byte of scratch before reading it.  Calls whose kernels may overlap on the
 * GPU (different streams with no ordering between them, or several host
 * threads) race on the array: issue them on one stream or synchronise
 * between them.
 *
 * Set-up: the first call on each device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and keeps it for later
 * calls; make that first call before any stream capture.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4k_matmul_tc_noalloc(const float *x, const void *w_q4k, float *y, int inputDim,
                          int outputDim, int tokens, q4mm_stream_t stream);

/* Bytes per row and 64-value chunk of the relayouted tensor-core layout, rows
 * per tile, and the size of a relayouted inputDim → outputDim weight (rows
 * rounded up to whole tiles). */
#define Q4MM_TC_CHUNK_BYTES 48
#define Q4MM_TC_TILE_ROWS 256
#define Q4MM_TC_RELAYOUT_BYTES(inputDim, outputDim)                                                \
    (((size_t)(outputDim) + Q4MM_TC_TILE_ROWS - 1) / Q4MM_TC_TILE_ROWS * Q4MM_TC_TILE_ROWS *        \
     (size_t)((inputDim) / 64) * Q4MM_TC_CHUNK_BYTES)

/*
 * q4k_relayout_tc — the one-time relayout of a Q4_K weight for
 * q4k_matmul_tc_relayouted: done once when the weight is registered, not on
 * every call (SKaiNET docs "Eager execution: backends and kernels", the
 * paragraph on weights relayouted once rather than per call; the page names
 * no target layout, so this one is the library's own).
 *
 * Layout written to w_tc.  Each 64-value chunk c of a row (values
 * 64c..64c+63: the slab j = c mod 4 of block b = c/4, its 32 code bytes
 * qs[32j..32j+31], low nibbles = sub-block 2j, high nibbles = 2j+1) becomes
 * 48 bytes:
 *   bytes  0..3  fp32 d·sc(2j)      bytes  4..7  fp32 dmin·m(2j)
 *   bytes  8..11 fp32 d·sc(2j+1)    bytes 12..15 fp32 dmin·m(2j+1)
 *   bytes 16..47 the 32 code bytes, unchanged
 * (floats little-endian).  Rows are grouped in tiles of Q4MM_TC_TILE_ROWS
 * (256), the last tile padded with zero rows, and stored tile-major: chunk c
 * of the 256 rows of tile t is one contiguous run of 256·48 bytes at byte
 * (t·(inputDim/64) + c)·12288, row r of the tile at 48·r within it.  The
 * tensor-core kernel then fetches each chunk of a tile with one plain bulk
 * copy.  Every product is exact in fp32, so the relayouted weight
 * dequantizes to the same fp32 matrix (w = scale·q − offset), and
 * q4k_matmul_tc_relayouted gives bit for bit the result of q4k_matmul_tc on
 * the canonical weight.  The layout keeps products, not factors: it cannot
 * be turned back into the canonical bytes.  It is about 4/3 the size of the
 * canonical weight (0.75·inputDim bytes per row, plus padding rows, against
 * 0.5625·inputDim).
 *
 * Arguments: w_q4k (device, read) the canonical weight, outputDim rows of
 * inputDim/256 blocks of 144 bytes; w_tc (device, written, padding rows
 * included) a buffer of Q4MM_TC_RELAYOUT_BYTES(inputDim, outputDim) bytes
 * owned by the caller.  Both 16-byte aligned, not overlapping; inputDim a
 * positive multiple of 256 up to Q4MM_MAX_INPUT_DIM, outputDim positive.
 * Asynchronous on `stream`; allocates nothing.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4k_relayout_tc(const void *w_q4k, void *w_tc, int inputDim, int outputDim, q4mm_stream_t stream);

/*
 * q4k_matmul_tc_relayouted — q4k_matmul_tc on a weight made by
 * q4k_relayout_tc: the same kernels, tiles, precision, scratch and results
 * (bit for bit); the dequantizing warps read the two sub-block scales of a
 * chunk as ready fp32 values instead of decoding the 6-bit scale field.
 * w_tc: Q4MM_TC_RELAYOUT_BYTES(inputDim, outputDim) bytes as q4k_relayout_tc
 * wrote them, 16-byte aligned.  Everything else as q4k_matmul_tc.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int q4k_matmul_tc_relayouted(const float *x, const void *w_tc, float *y, int inputDim, int outputDim,
                             int tokens, q4mm_stream_t stream);

/*
 * ternary_gemv — y = scale · (x·codesᵀ) with W in the BitNet b1.58 payload.
 *
 * Defined by SKaiNET issue #1138 "[ternary-f32] Phase 2: TernaryF32GemvNative
 * SPI + reference ViewKernel + TernaryF32KernelPack", section "Tasks": four
 * codes per byte, code(o, i) = ((byte >> 2·(i%4)) & 3) − 1 for byte
 * o·K/4 + i/4; out[o] = Σ_k in[k]·code(o,k) accumulated in FP32; the scale
 * multiplies the finished dot product once (pass 1.0f for the seam's raw,
 * unscaled code-dot); rows for prefill advance by r·k and r·n.
 *
 * w_packed : N rows of K/4 bytes, no alignment required.  x: 16-byte
 *            aligned.  y: 4-byte aligned.
 * Limits: inputDim a positive multiple of 4 and <= Q4MM_MAX_INPUT_DIM;
 *         outputDim >= 1; tokens >= 1.
 * Precision: FP32.  The field value 3 decodes to +2 by the literal formula.
 *            With integer activations the code-dot is exact, so y equals
 *            the single fp32 rounding of scale × dot bit for bit.  Up to 3
 *            tokens with inputDim a multiple of 256 (and W 16-byte aligned)
 *            x is split as in q4k_matmul's one-token path and the code-dot
 *            is an exact integer sum of code·x̂.
 * Returns Q4MM_OK or Q4MM_ERR_{DIM,NULL,ALIGN,ALIAS,CUDA}.
 */
int ternary_gemv(const float *x, const void *w_packed, float scale, float *y, int inputDim,
                 int outputDim, int tokens, q4mm_stream_t stream);

/* Message for the last error returned on the calling thread ("" if none).
 * The pointer stays valid until the thread's next failing call. */
const char *q4mm_last_error(void);

/*
 * q4mm_device_status — waits for `stream`, then returns Q4MM_OK, or
 * Q4MM_ERR_TIMEOUT if a bounded in-kernel wait of an earlier call on the
 * current device ran out.  clear != 0 resets the status word afterwards.
 * Returns Q4MM_ERR_CUDA if the stream reports an error.
 */
int q4mm_device_status(q4mm_stream_t stream, int clear);

/*
 * q4mm_test_fail_next_wait — a test hook for the library's failure
 * detection; the pages have no counterpart.  The calling thread's next call
 * of q4k_matmul (one-token and 3-8 token kernels), q4_0_gemv, q6k_gemv,
 * q4k_ffn_swiglu or q4k_matmul_tc never issues the copy of weight stage
 * `stage` of each CTA (its ring stage, or its 256-row weight tile on the
 * tensor cores) and bounds every in-kernel wait by `limit_cycles` SM cycles
 * (about 2·10^6 per millisecond) instead of about 2·10^9.  The waits on the
 * missing stage then run out: the kernel sets the device status word, lets
 * every copy it did issue land, and exits; that call's y is undefined and
 * q4mm_device_status reports Q4MM_ERR_TIMEOUT.  Nothing faults or waits
 * without a bound.  Later calls, and calls on other threads, are not
 * affected; a call rejected by validation leaves it armed.  stage = -1
 * disarms it; otherwise stage >= 0 and limit_cycles > 0, else Q4MM_ERR_DIM.
 */
int q4mm_test_fail_next_wait(int stage, long long limit_cycles);

/* Library version, major·10000 + minor·100 + patch. */
int q4mm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q4MM_H */
