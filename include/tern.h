/*
 * tern.h -- C ABI of the B300 ternary packed-weight linear layer.
 *
 * The operation (Neutrino-1 8B model page: the intro states that all 252
 * transformer linears use a ternary-family weight format kept bit-packed in
 * memory and decoded by the matrix kernels themselves; "Where the bytes
 * live" lists per-row metadata of row dimensions, scales and row sums) is,
 * for one projection with R output rows and K inputs,
 *
 *     y[m][r] = scale[r] * sum_{k < K} t[r][k] * x[m][k],   t[r][k] in {-1,0,+1}
 *
 * with the ternary matrix t kept in a 2-bit packed form and decoded inside the
 * kernels (never expanded to a floating-point weight tensor in memory).
 *
 * Packed format.  The page calls its own format proprietary and never
 * describes its bits, so this library fixes its own:
 *   - K must be a multiple of 64 (pad rows with zero weights);
 *   - codes: R * K/16 uint32 words, row-major and K-contiguous; row r owns
 *     words [r*K/16, (r+1)*K/16) (16-byte aligned rows);
 *   - column k of a row sits in word k/16 of that row at bits 2*(k%16) (b0,
 *     low) and 2*(k%16)+1 (b1, high): least significant code first;
 *   - (b1,b0): 00 -> 0, 01 -> +1, 11 -> -1 (2-bit two's complement);
 *     10 is invalid: tern_pack never writes it, tern_validate reports it, and
 *     the device kernels give an unspecified (but fault-free) result for it;
 *   - scale: R fp32, applied after the sum;
 *   - rowsum: R int32, rowsum[r] = sum_k t[r][k] (validation and closed-form
 *     checks; the GEMV kernels do not read it).
 *
 * Activations x are bf16, passed as their uint16 bit patterns, row-major
 * [M][K] (M = 1 for the GEMV), finite.  Outputs are fp32, row-major [M][R].
 *
 * Arithmetic.  The kernels decode each code to an e4m3 weight of exactly
 * 0 or +-2 and multiply on the tensor cores with fp32 accumulation.  Each
 * activation row enters as e4m3 terms under power-of-two scales, per row
 * and per K range a kernel stages at once (a chunk): x = (hi + lo/16) * 2^-s
 * with hi, lo e4m3, which is exact for every element at least 2^-13 of the
 * row's maximum (2^e <= max|x| < 2^(e+1)) and off by at most 2^(e-21)
 * below that.  When those smaller elements could move the row's sum by more
 * than 2^-24 of sum|x| (n_small * 2^(e-21) > 2^-24 * sum|x|: outlier
 * channels), the chunk is taken in two bands instead: band A holds the
 * elements within 2^13 of the maximum, band B the others under a scale of
 * their own (2^f <= band-B max < 2^(f+1)), exact down to 2^-13 of it and
 * off by at most 2^(f-21) below.  Within a band the sums are fp32; bands
 * and split-K ranks are added as exact fp32 pairs (TwoSum) and rounded
 * once.  The batched kernel adds a unit's chunks in plain fp32 while every
 * chunk so far has had one band (each is then within 2^-24 of its own
 * sum|x|), and as pairs from the unit's first two-band chunk on.
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer it passes.  Device memory the library
 *     holds itself: one error word per kernel family and the
 *     TERN_NOALLOC_WS_BYTES array of tern_gemm_batched_noalloc (both
 *     module-scope, set up when the library's kernels are loaded on a
 *     device), and the workspaces tern_gemm_batched (and _rmsnorm) and
 *     tern_lmhead_argmax allocate on first need (see there).  tern_gemv,
 *     tern_gemv_swiglu, tern_gemm_smallm*, tern_unpack and
 *     tern_gemm_batched_noalloc never allocate.
 *   - Encoded TMA descriptors of weight matrices are cached on the host by
 *     (codes pointer, shape); a descriptor holds only that address and
 *     shape, so a later matrix at the same address with the same shape
 *     reuses it correctly.
 *   - Device entry points are asynchronous on the caller's stream
 *     (a cudaStream_t passed as void*; NULL is the legacy default stream).
 *     Arguments are checked on the host before anything is launched; a
 *     failed check returns an error and launches nothing.
 *   - No C++ exception crosses this boundary.
 *   - A problem with rows == 0 is empty: it succeeds without a launch and its
 *     pointers may be NULL.  K == 0 is valid and gives y = 0.
 */
#ifndef TERN_H
#define TERN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TERN_ABI_VERSION 2

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define TERN_API __attribute__((visibility("default")))
#else
#define TERN_API
#endif

/* Largest activation block the device kernels stage on chip:
 * m * k * 2 bytes (bf16) must not exceed this. */
#define TERN_MAX_X_BYTES 196608
/* Largest activation row count of tern_gemm_smallm*. */
#define TERN_MAX_M 8
/* Size of the fixed scratch of tern_gemm_batched_noalloc (4 MiB). */
#define TERN_NOALLOC_WS_BYTES 4194304

typedef enum {
    TERN_OK = 0,
    TERN_ERR_NULL = 1,    /* a required pointer is NULL */
    TERN_ERR_SHAPE = 2,   /* rows/k negative, k % 64 != 0, size limits, shape mismatch */
    TERN_ERR_ALIGN = 3,   /* a pointer breaks its alignment rule */
    TERN_ERR_BADCODE = 4, /* packed data holds the invalid pattern 10 */
    TERN_ERR_ROWSUM = 5,  /* stored rowsum disagrees with the codes */
    TERN_ERR_M_RANGE = 6, /* m outside [1, TERN_MAX_M] */
    TERN_ERR_CUDA = 7,    /* a CUDA runtime call or launch failed */
    TERN_ERR_TIMEOUT = 8, /* a device-side bounded wait ran out (see tern_last_device_error) */
    TERN_ERR_VALUE = 9    /* a value outside its range: an int8 weight given to tern_pack that is
                             not -1, 0 or +1, or an RMSNorm eps that is negative or not finite */
} tern_status;

/* One packed ternary matrix.  Pointers are device pointers for the device
 * entry points.  codes: 16-byte aligned.  scale: 4-byte aligned.  rowsum:
 * may be NULL (not read by the device kernels). */
typedef struct {
    int32_t rows;           /* R >= 0 */
    int32_t k;              /* K >= 0, K % 64 == 0 */
    const uint32_t *codes;  /* R * K/16 words */
    const float *scale;     /* R */
    const int32_t *rowsum;  /* R, or NULL */
} tern_matrix;

/* ---------------------------------------------------------------------- */
/* Host-side packer and validator (host memory, synchronous).              */
/* ---------------------------------------------------------------------- */

/* Pack an int8 matrix t [rows][k] (values -1, 0, +1) into codes
 * [rows][k/16] and write rowsum[rows] (rowsum may be NULL).
 * The per-row metadata follows "Where the bytes live" (scales and row sums).
 * Errors: TERN_ERR_NULL, TERN_ERR_SHAPE (k % 64, negative sizes),
 * TERN_ERR_VALUE (a weight outside {-1,0,+1}; codes are then incomplete). */
TERN_API tern_status tern_pack(const int8_t *t, int32_t rows, int32_t k,
                      uint32_t *codes, int32_t *rowsum);

/* Check packed codes: no invalid pattern, and (if rowsum != NULL) every
 * stored rowsum equals the sum of its row.  counts_out (may be NULL) receives
 * {zeros, plus ones, minus ones} over the whole matrix: the statistics the
 * model page reports in "Inside the coded lane".
 * Errors: TERN_ERR_NULL, TERN_ERR_SHAPE, TERN_ERR_BADCODE (first bad word
 * stops the scan; counts are then partial), TERN_ERR_ROWSUM. */
TERN_API tern_status tern_validate(const uint32_t *codes, int32_t rows, int32_t k,
                          const int32_t *rowsum, int64_t counts_out[3]);

/* ---------------------------------------------------------------------- */
/* Device entry points (device pointers, asynchronous on `stream`).        */
/* ---------------------------------------------------------------------- */

/* Decode a packed matrix to int8 t_out [rows][k] (debug / exactness gate;
 * the in-kernel decode made visible).  t_out: 16-byte aligned.
 * The invalid pattern decodes to -2. */
TERN_API tern_status tern_unpack(const tern_matrix *w, int8_t *t_out, void *stream);

/* M = 1 decode-time GEMV: y[r] = scale[r] * sum_k t[r][k] x[k].
 * x: k bf16 values, 16-byte aligned.  y: rows fp32, 4-byte aligned.
 * x and y must not overlap the matrix.  Limit: 2*k <= TERN_MAX_X_BYTES. */
TERN_API tern_status tern_gemv(const tern_matrix *w, const uint16_t *x, float *y, void *stream);

/* Fused gated feed-forward pair (spec table: gated SwiGLU feed-forward,
 * three linears per layer): h[r] = silu(g[r]) * u[r] with
 * g = gate projection of x, u = up projection of x, silu(z) = z/(1+exp(-z)).
 * gate and up must have equal rows and k.  h: rows fp32. */
TERN_API tern_status tern_gemv_swiglu(const tern_matrix *gate, const tern_matrix *up,
                             const uint16_t *x, float *h, void *stream);

/* Small-M GEMM for speculative verification (the page's verifier scores a
 * six-token draft plus one token in one forward pass, so M = 7):
 * y[i][r] = scale[r] * sum_k t[r][k] x[i][k] for i < m, 1 <= m <= TERN_MAX_M.
 * x: [m][k] bf16, 16-byte aligned.  y: [m][rows] fp32.
 * Errors add TERN_ERR_M_RANGE.  Limit: m*k*2 <= TERN_MAX_X_BYTES. */
TERN_API tern_status tern_gemm_smallm(const tern_matrix *w, const uint16_t *x, int32_t m,
                             float *y, void *stream);

/* Small-M fused gate/up: h[i][r] = silu(g[i][r]) * u[i][r], i < m. */
TERN_API tern_status tern_gemm_smallm_swiglu(const tern_matrix *gate, const tern_matrix *up,
                                    const uint16_t *x, int32_t m, float *h, void *stream);

/* One item of a batched call: y = W x when up == NULL, or the fused pair
 * h = silu(W x) * (up x) (W is then the gate), for m activation rows.
 * Pointers and layouts as for the single calls above. */
typedef struct {
    const tern_matrix *w;   /* weights (the gate of a SwiGLU pair) */
    const tern_matrix *up;  /* NULL, or the up projection of a SwiGLU pair */
    const uint16_t *x;      /* [m][k] bf16, 16-byte aligned */
    float *y;               /* [m][rows] fp32 */
    int32_t m;              /* 1 <= m <= TERN_MAX_M */
} tern_batch_item;

/* Many independent products in one persistent launch (one CTA per SM
 * streaming a byte-balanced share of all items' weights): the seven linears
 * of a layer, the 252 linears of a token, a batch of projections.  Items
 * must be independent: no item's y may overlap another item's x, y or
 * weights.  Every item is checked as by the single calls before anything is
 * launched; the first failing item's status is returned and nothing runs.
 * Items are launched in order on `stream` in groups of consecutive items:
 * a launch takes up to 128 items holding up to 144 weight matrices (a SwiGLU
 * pair holds two), and a batch that needs several launches is spread evenly
 * over the fewest that fit; an item with k == 0 (y = 0) takes a small launch
 * of its own and one with rows == 0 none.  Tensor maps of the weights are
 * encoded once per (codes, shape) and cached by the library, so repeated
 * calls on resident weights cost a lookup on the host.
 * Workspace: when a launch group holds items with m >= 2, a short kernel
 * runs just before it and writes those items' activations, split into the
 * operand form the tensor cores read, to a device workspace that the library
 * owns: one per (context, stream), allocated with cudaMalloc on first need
 * (also while the stream is being captured), grown by doubling and never
 * freed, since a captured launch keeps its address.  Launches on one stream
 * are ordered, so they share it safely; a captured graph must not run at the
 * same time as other calls on the stream it was captured on.  If the
 * allocation fails the call returns TERN_ERR_CUDA (launch groups before the
 * failing one have been launched); tern_gemm_batched_noalloc needs no
 * allocation.  n == 0 is a no-op; items == NULL gives TERN_ERR_NULL, n < 0
 * TERN_ERR_SHAPE. */
TERN_API tern_status tern_gemm_batched(const tern_batch_item *items, int32_t n, void *stream);

/* Number of kernel launches tern_gemm_batched makes for these items (host
 * only, nothing is launched and only items[i].w->rows and ->k are read; the
 * items are not otherwise checked), counting the activation-preparing
 * launch of each group that holds items with m >= 2.  0 for n == 0; a
 * negative tern_status for
 * n < 0 (-TERN_ERR_SHAPE) or a NULL items array or weight pointer
 * (-TERN_ERR_NULL).  Not an operation of the model pages: a planning aid for
 * callers that count or capture launches. */
TERN_API int32_t tern_gemm_batched_launches(const tern_batch_item *items, int32_t n);

/* tern_gemm_batched with an RMSNorm ahead of each item's projection (model
 * page spec table: RMSNorm with eps 1e-6 before the attention and
 * feed-forward blocks, whose first linears are q/k/v and gate/up).  For an
 * item i with norm_w[i] != NULL, each activation row x[j] is first replaced
 * by xn[j][c] = bf16_rn(norm_w[i][c] * fl32(x[j][c] * r_j)), with
 * r_j = fl32(1 / sqrt(mean_c x[j][c]^2 + eps)) (mean over the item's k
 * channels, taken in fp64; eps widened to fp64): the page gives only the
 * textbook operation, and this library rounds the normalised activations to
 * bf16 because the projection consumes bf16.  Items with norm_w[i] == NULL
 * run as in tern_gemm_batched.  x itself is not modified.
 * norm_w: host array of n pointers; each non-NULL entry is a device array of
 * the item's k fp32 channel weights, 16-byte aligned.  eps: finite, >= 0.
 * Launches, workspace and checks are those of tern_gemm_batched, plus
 * TERN_ERR_NULL (norm_w == NULL with n > 0), TERN_ERR_VALUE (eps negative,
 * NaN or infinite) and TERN_ERR_ALIGN (a misaligned norm_w[i]).
 * Accuracy: r_j is rounded from an fp64 sum whose order is the kernel's own,
 * so in rare rows it may differ from a sequential sum's by one fp32 ulp;
 * everything else is fixed above. */
TERN_API tern_status tern_gemm_batched_rmsnorm(const tern_batch_item *items, const float *const *norm_w,
                                               float eps, int32_t n, void *stream);

/* tern_gemm_batched for callers that must not allocate device memory: code
 * running inside a memory budget that another allocator owns (a serving
 * engine that reserves the GPU's memory for its caches up front, where a
 * cudaMalloc from the library may fail or fragment that pool), and code
 * that may not call cudaMalloc at all.  The model pages have no counterpart:
 * the operation, items, checks, launches and results are those of
 * tern_gemm_batched, byte for byte.  The difference is where the prepared
 * activations of items with m >= 2 live: a module-scope device array of
 * TERN_NOALLOC_WS_BYTES, set up by the CUDA runtime with the library's
 * kernels, instead of the per-stream workspace.
 * Limit: every launch group's prepared activations (about m * k * 4 bytes per
 * item with m >= 2, k padded to a multiple of 512) must fit the array; a batch
 * that needs more gets TERN_ERR_SHAPE before anything is launched.
 * The array takes its device memory when the CUDA runtime loads the
 * library's kernels on a device, which with lazy module loading (the
 * default) is the first launch of this file's kernels there, possibly this
 * call: make one warm-up call (n == 1, one small item) on each device
 * before reserving the device's memory for other pools and before
 * capturing a stream.  The first call in a context also looks the array's
 * address up (cudaGetSymbolAddress, with that device current;
 * TERN_ERR_CUDA if that fails); a context created after a device reset
 * looks it up again.  Nothing in the array must start at zero: each launch
 * writes every byte it reads.  There is one array per device, shared by
 * every stream: calls whose launches overlap in time (on different
 * streams, or a captured graph replayed beside another call) race on it. */
TERN_API tern_status tern_gemm_batched_noalloc(const tern_batch_item *items, int32_t n, void *stream);

/* An int8 matrix with per-row scales: the output head of the model page
 * ("Where the bytes live": a 151,936 x 4,096 int8 head, scaled per row).
 * w: rows * k int8, row-major, 16-byte aligned; scale: rows fp32. */
typedef struct {
    int32_t rows;        /* R >= 1 */
    int32_t k;           /* K >= 64, K % 64 == 0 */
    const int8_t *w;     /* R * K */
    const float *scale;  /* R */
} tern_i8_matrix;

/* Output head with the greedy choice fused (model page: the int8 head, read
 * once per generated token, and the speculative verifier's greedy
 * acceptance): for each activation row i < m,
 *     logits[i][r] = scale[r] * sum_k w[r][k] * x[i][k]      (fp32)
 *     argmax[i]    = the r of the largest logits[i][r], the lowest r on ties,
 * where the argmax is taken over the fp32 logits this call writes.  With
 * norm_w != NULL each x row is first normalised as in
 * tern_gemm_batched_rmsnorm (the final norm ahead of the head).
 * x: [m][k] bf16, 16-byte aligned; logits: [m][rows] fp32, 4-byte aligned;
 * argmax: m int32, 4-byte aligned; norm_w: NULL or k fp32, 16-byte aligned.
 * 1 <= m <= TERN_MAX_M, m * k * 2 <= TERN_MAX_X_BYTES.
 * Arithmetic: each weight enters the tensor cores as two exact e4m3 nibble
 * terms and x as e4m3 terms as in the ternary products, so the logits are
 * fp32 sums of exact products; their error is a few fp32 roundings of
 * sum_k |w x| (not of the logit itself).
 * Launches: a 1-thread-block kernel that resets the argmax state, the
 * activation-preparing kernel when m >= 2, the persistent kernel, and a
 * 1-thread-block kernel that writes argmax.  Workspace: as tern_gemm_batched,
 * plus 64 bytes per (context, stream) for the argmax state.
 * Errors: TERN_ERR_NULL, TERN_ERR_SHAPE (rows < 1, k < 64, k % 64, m * k * 2
 * over the limit), TERN_ERR_M_RANGE, TERN_ERR_ALIGN, TERN_ERR_VALUE (eps),
 * TERN_ERR_CUDA. */
TERN_API tern_status tern_lmhead_argmax(const tern_i8_matrix *w, const uint16_t *x, int32_t m,
                                        const float *norm_w, float eps, float *logits, int32_t *argmax,
                                        void *stream);

/* A denser packing: five ternary weights per byte, 1.6 bits a weight (the
 * model page's byte budget, "Where the bytes live", spends more bits per
 * weight than a ternary value needs; this format is the library's own):
 *   - K must be a multiple of 80 (pad rows with zero weights);
 *   - codes: R * K/5 bytes, row-major; byte j of a row holds weights
 *     5j .. 5j+4 as b = sum_{i<5} (t_{5j+i} + 1) * 3^i (least significant
 *     digit first), b in [0, 242]; 243..255 are invalid: tern5_pack never
 *     writes them and the device kernels give an unspecified (but fault-free)
 *     result for them (tern5_unpack writes -2);
 *   - scale: R fp32, applied after the sum.
 * codes: 16-byte aligned; scale: 4-byte aligned. */
typedef struct {
    int32_t rows;          /* R >= 0 */
    int32_t k;             /* K >= 0, K % 80 == 0 */
    const uint8_t *codes;  /* R * K/5 */
    const float *scale;    /* R */
} tern5_matrix;

/* Pack an int8 matrix t [rows][k] (values -1, 0, +1; k % 80 == 0) into
 * base-3 codes [rows][k/5] and write rowsum[rows] (may be NULL).  Host
 * memory, synchronous.  Errors: TERN_ERR_NULL, TERN_ERR_SHAPE,
 * TERN_ERR_VALUE. */
TERN_API tern_status tern5_pack(const int8_t *t, int32_t rows, int32_t k, uint8_t *codes, int32_t *rowsum);

/* Decode base-3 codes to int8 t_out [rows][k] on the device (bit-exact). */
TERN_API tern_status tern5_unpack(const tern5_matrix *w, int8_t *t_out, void *stream);

/* y[i][r] = scale[r] * sum_k t[r][k] x[i][k], i < m, from base-3 codes, on
 * the CUDA cores (each byte's five digits by division by 3 as a multiply
 * and shift; fp32 accumulation).  x: [m][k] bf16, 16-byte aligned; y:
 * [m][rows] fp32.  1 <= m <= TERN_MAX_M, m * k * 2 <= TERN_MAX_X_BYTES.
 * One launch; allocates nothing.  Errors as tern_gemm_smallm. */
TERN_API tern_status tern5_gemm(const tern5_matrix *w, const uint16_t *x, int32_t m, float *y, void *stream);

/* Synchronise `stream`, then report and clear the device error word that
 * bounded device-side waits set when they run out (TERN_ERR_TIMEOUT), or a
 * pending CUDA error (TERN_ERR_CUDA).  TERN_OK otherwise. */
TERN_API tern_status tern_last_device_error(void *stream);

/* Bound of every device-side mbarrier wait of later launches, in SM clock
 * cycles (default 2^31, about one second at the B300's maximum clock);
 * cycles <= 0 restores the default.  A wait that runs out sets the device
 * error word, and the kernel stops, waits (with the default bound) for its
 * own copies and MMAs in flight, releases its tensor memory and returns, so
 * the context stays usable and tern_last_device_error reports
 * TERN_ERR_TIMEOUT.  Not an operation of the model pages: a diagnostic that
 * lets a test make a wait run out.  Launches already made, and launches
 * captured in a graph, keep the bound they were made with. */
TERN_API void tern_set_wait_limit(int64_t cycles);

/* Static description of a status code (never NULL). */
TERN_API const char *tern_status_str(tern_status s);

/* TERN_ABI_VERSION of the loaded library. */
TERN_API int32_t tern_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TERN_H */
