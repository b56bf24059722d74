/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA recurrent-state library.
 *
 * Kimi Delta Attention (KDA) keeps, per layer, request slot and value head, a
 * recurrent state S of shape [K][V] (V innermost).  At decode and at
 * speculative verify each token applies the fused sigmoid-gated delta rule
 *
 *     khat = k / sqrt(sum k^2 + 1e-6),  qhat = q / sqrt(sum q^2 + 1e-6)
 *     beta = sigmoid(b),                alpha_i = exp(-softplus(a_i))
 *     S <- diag(alpha) S;   u = S^T khat;   S <- S + beta khat (v - u)^T
 *     o = S^T qhat / sqrt(K)
 *
 * (ROCm/ATOM pull request 2130, "perf(kimi-k3): make the KDA temporal state
 * dtype configurable", What: the [12,128,128] state, q and k normalised in the
 * kernel, fused sigmoid gating; ROCm/ATOM pull request 2945, Summary and
 * Changes: the state pool's dtype is a build constant, a loaded fp16 state is
 * widened to fp32, the recurrence runs in fp32, a stored state is rounded to
 * fp16 to nearest even, and every state access goes through one address
 * function state_at(c, slot).)
 *
 * One library file is built per pool dtype: libkda_h0.so (fp32 pool) and
 * libkda_h1.so (fp16 pool), after the _h0/_h1 kernel names of pull request
 * 2945 (Changes).  A pool of the other dtype is refused at call time.
 *
 * Conventions for every entry point:
 *  - Return value: KDA_OK (0) or a kda_status code; argument errors are
 *    detected on the host, synchronously, before anything is launched.
 *  - Memory: the caller owns every buffer and the stream; no call allocates
 *    memory, keeps state between calls or synchronises.  One exception to
 *    "the library holds no memory": each library build carries the
 *    KDA_PREFILL_SCRATCH_BYTES (128 MB) scratch array of
 *    kda_prefill_chunked_noalloc as a file-scope device array, resident on
 *    every device where the library's module is loaded (by its first kernel
 *    launch of any kind) for the life of the process, whether or not that
 *    entry point is ever called; a process that loads both builds holds
 *    256 MB per device.  Pointers marked "device" must be device-accessible
 *    (cudaMalloc'd); pointers marked "host" are read on the host during the
 *    call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; outputs are valid once it completes.
 *  - Device-side errors do not trap.  A slot id outside [0, num_slots): the
 *    affected (request, head) tiles are skipped and KDA_ERR_SLOT_RANGE is
 *    written to *dev_status (first error wins).  A pipeline wait inside the
 *    kernel that has not completed after 1 s: KDA_ERR_TIMEOUT is written and
 *    the kernel drains its copies and exits.  The caller zeroes *dev_status
 *    before the call and reads it after synchronising.
 *  - Preconditions not checked on the hot path: the slot ids of different
 *    requests (and the snapshot slots of one call) are pairwise distinct, and
 *    no other work touches those slots while the call runs.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_dtype {
    KDA_F32 = 0,   /* IEEE binary32 */
    KDA_F16 = 1,   /* IEEE binary16 */
    KDA_BF16 = 2   /* bfloat16: accepted for q/k/v, refused for a state pool */
} kda_dtype;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,              /* a required pointer is NULL */
    KDA_ERR_DTYPE_MISMATCH = 2,    /* pool dtype is not this library's build dtype */
    KDA_ERR_DTYPE_UNSUPPORTED = 3, /* pool dtype other than fp32/fp16 (bf16 included), or a bad q/k/v dtype */
    KDA_ERR_LAYERS_DISAGREE = 4,   /* kda_pool_check: layers differ in dtype or shape */
    KDA_ERR_SHAPE = 5,             /* K or V outside 16..128 or not a multiple of 16; bad counts or strides */
    KDA_ERR_ALIGN = 6,             /* pool base, slot stride, q, k, v or a not 16-byte aligned; b, o, ids not 4-byte */
    KDA_ERR_LAUNCH = 7,            /* the CUDA launch itself failed */
    KDA_ERR_SLOT_RANGE = 8,        /* device: a slot id outside [0, num_slots); its tiles were skipped */
    KDA_ERR_ARG = 9,               /* any other bad argument (negative counts, n_layers < 1) */
    KDA_ERR_TIMEOUT = 10,          /* device: a pipeline wait gave up after 1 s; results incomplete */
    KDA_ERR_LAYOUT = 11            /* a checkpoint plane written under another state layout (dtype or shape) */
} kda_status;

/*
 * Launch options of kda_decode_step and kda_spec_verify (bitwise OR; 0 = none).
 *
 * KDA_LAUNCH_PDL: launch with programmatic stream serialization, so the kernel
 *   may be scheduled while the previous kernel on the stream is still running
 *   (it starts its set-up there).  It reads and writes nothing the previous
 *   kernel may write until that kernel has completed.  Without a previous
 *   kernel on the stream this has no effect.
 * KDA_LAUNCH_PDL_EARLY_STATE: with KDA_LAUNCH_PDL, the kernel also reads the
 *   slot ids, reset flags and its first state tiles before the previous kernel
 *   has completed, so the state stream overlaps that kernel's tail.  Only valid
 *   when the previous kernel on the stream writes none of those: e.g. it is a
 *   projection producing q/k/v/a/b, or a step on another layer's pool.  Two
 *   back-to-back calls on the same pool must not use it.  For kda_conv_step
 *   the early reads are the token offsets, slot ids, accepted indices, reset
 *   flags, weights, bias and the window entries; x is read, and y and the
 *   window are written, only after the previous kernel has completed.
 */
#define KDA_LAUNCH_PDL 1u
#define KDA_LAUNCH_PDL_EARLY_STATE 2u

/*
 * KDA_LAUNCH_TEST_WITHHOLD_STATE: a test hook of kda_decode_step,
 *   kda_spec_verify and kda_step, for the timeout path only; never for
 *   production calls, and refused by every other entry point.  Each tile arms
 *   its state tile's barrier but withholds the copy, so every wait on it gives
 *   up at its 1 s bound: the call then reports KDA_ERR_TIMEOUT through
 *   dev_status (after about 2 s: the wait, then a bounded drain), writes
 *   neither those tiles' states nor their outputs, and the context stays
 *   usable.  Requests that reset (no state read) are not affected.
 */
#define KDA_LAUNCH_TEST_WITHHOLD_STATE (1u << 30)

/*
 * One layer's state pool: num_slots slots, each holding hv heads of a [k][v]
 * state (v innermost, row-major), all in device memory.
 *   state_at(slot, h) = base + (slot * slot_stride + h * k * v) elements.
 * slot_stride is in elements and must be >= hv * k * v (pass hv * k * v for a
 * dense pool); slot_stride * element size must be a multiple of 16 bytes and
 * base must be 16-byte aligned (the kernels move the state in 16-byte vectors).
 */
typedef struct kda_pool {
    void* base;           /* device */
    int32_t dtype;        /* kda_dtype: KDA_F32 or KDA_F16 */
    int32_t hv;           /* value heads per slot */
    int32_t k;            /* key dimension K: 16..128, multiple of 16 */
    int32_t v;            /* value dimension V: 16..128, multiple of 16 */
    int64_t num_slots;    /* slots in the pool */
    int64_t slot_stride;  /* elements from one slot to the next */
} kda_pool;

/* The pool dtype this library was built for: KDA_F32 (libkda_h0) or KDA_F16
 * (libkda_h1).  (Pull request 2945, Changes: the dtype is a build-key field.) */
int kda_build_state_dtype(void);

/*
 * Host-only check of the pools of n_layers layers (no device access): every
 * pool is fp32 or fp16 (else KDA_ERR_DTYPE_UNSUPPORTED), all layers share one
 * dtype, hv, k and v (else KDA_ERR_LAYERS_DISAGREE), that dtype is this
 * build's (else KDA_ERR_DTYPE_MISMATCH), and each pool's shape and alignment
 * are valid (KDA_ERR_SHAPE / KDA_ERR_ALIGN / KDA_ERR_NULL).
 * (Pull request 2945, Changes: one recurrent dtype across every layer; a step
 * refuses a pool of the other dtype; only fp32 or fp16 are accepted because
 * anything else would be reinterpreted rather than converted.)
 * pools: host array [n_layers].
 */
int kda_pool_check(const kda_pool* pools, int32_t n_layers);

/*
 * Host-only: the bytes of state one slot of `pool` holds (hv * k * v * element
 * size) in *bytes_per_slot (host).  Returns KDA_ERR_DTYPE_UNSUPPORTED for a
 * dtype other than fp32/fp16.  (Pull request 2130, Memory: the per-slot state
 * size scales with the element size.)
 */
int kda_state_bytes(const kda_pool* pool, int64_t* bytes_per_slot);

/*
 * One decode token for each of n requests, all value heads.  The state of
 * request r is read from slot slot_ids[r] (or taken as zero when reset[r] is
 * nonzero), updated, and written back in place to the same slot.
 *   pool      host pointer to the descriptor; the pool memory is device.
 *   slot_ids  device int32 [n].
 *   reset     device uint8 [n], or NULL for "no request resets".
 *   q, k      device [n][hv][k] of qkv_dtype (KDA_F32, KDA_F16 or KDA_BF16).
 *   v         device [n][hv][v] of qkv_dtype.
 *   a         device fp32 [n][hv][k]: decay logits; alpha = exp(-softplus(a)).
 *             q, k, v and a must be 16-byte aligned (they move by bulk copy).
 *   b         device fp32 [n][hv]: beta logits; beta = sigmoid(b).
 *   o         device fp32 [n][hv][v] (output).
 *   dev_status device int32 [1]; the caller zeroes it; see conventions.
 *   flags     KDA_LAUNCH_* bits (unknown bits: KDA_ERR_ARG).
 *   stream    cudaStream_t to enqueue on (NULL: the legacy default stream).
 * n == 0 is a no-op returning KDA_OK after the pool checks (buffers may then be NULL).
 */
int kda_decode_step(const kda_pool* pool, const int32_t* slot_ids, const uint8_t* reset,
                    int32_t n, const void* q, const void* k, const void* v,
                    int32_t qkv_dtype, const float* a, const float* b, float* o,
                    int32_t* dev_status, uint32_t flags, void* stream);

/*
 * Speculative verify: t tokens per request (the accepted token and the draft
 * tokens), applied one after another.  The state of request r is read once
 * from init_slot[r] (or zero when reset[r] is nonzero), carried in fp32
 * between tokens without rounding, and after token j it is stored (rounded to
 * the pool's dtype) to snapshot slot snap_slot[r][j].  init_slot[r] itself is
 * not written unless it is also one of the snapshot slots.
 * (Pull request 2945, Changes: state_at serves each token's snapshot slot.)
 *   init_slot device int32 [n];  snap_slot device int32 [n][t].
 *   q, k      device [n][t][hv][k] of qkv_dtype;  v device [n][t][hv][v].
 *   a         device fp32 [n][t][hv][k];  b device fp32 [n][t][hv].
 *   o         device fp32 [n][t][hv][v] (output).
 * Other arguments as for kda_decode_step.  n == 0 or t == 0 is a no-op
 * returning KDA_OK after the pool checks (buffers may then be NULL).
 */
int kda_spec_verify(const kda_pool* pool, const int32_t* init_slot, const int32_t* snap_slot,
                    const uint8_t* reset, int32_t n, int32_t t, const void* q,
                    const void* k, const void* v, int32_t qkv_dtype, const float* a,
                    const float* b, float* o, int32_t* dev_status, uint32_t flags,
                    void* stream);

/*
 * Arguments of kda_step, the general step.  Pointers are device pointers
 * unless noted; the optional ones may be NULL.
 *
 * Request r owns tokens cu_seqlens[r] .. cu_seqlens[r+1] - 1 of the packed
 * inputs (T_r of them, 0 <= T_r <= max_t), or, with cu_seqlens NULL, tokens
 * r * max_t .. r * max_t + max_t - 1.  Its row of slot_table holds num_cols
 * slots: state_at(c, slot) of pull request 2945, Changes -- one address
 * function for a request's initial state and for each token's snapshot.  The
 * initial state is read from column accepted[r] - 1 (column 0 when accepted
 * is NULL), so a step starts from the snapshot of the last token the previous
 * step accepted; the state after token j is stored to column j.  A negative
 * initial slot marks a padding request: nothing is read or stored and its
 * output rows are zero.  A negative snapshot slot means that token's state is
 * not kept (the recurrence still runs through it).
 * in_place != 0 is decode: one token per request (cu_seqlens NULL, total == n,
 * max_t == 1), the state stored back to the initial slot (the decode kernel).
 *
 * Heads: q and k have h_qk heads and value head h reads q/k head
 * h / (hv / h_qk) (hv % h_qk == 0; h_qk == hv is one q/k per value head).
 * Gate: alpha = exp(-softplus(a)) without a_log; with a_log,
 * alpha = exp(-exp(a_log[h]) * softplus(a + dt_bias[h])) (dt_bias NULL: 0).
 */
typedef struct kda_step_args {
    int32_t n;                  /* requests */
    int32_t total;              /* packed tokens: rows of q, k, v, a, b, o */
    int32_t max_t;              /* most tokens of any request; <= num_cols unless in_place */
    int32_t h_qk;               /* q/k heads */
    int32_t num_cols;           /* columns of slot_table (>= 1) */
    int32_t in_place;           /* 0: speculative step; nonzero: decode in place */
    int32_t qkv_dtype;          /* KDA_F32, KDA_F16 or KDA_BF16 */
    int32_t reserved;           /* 0 */
    const int32_t* cu_seqlens;  /* [n + 1] or NULL */
    const int32_t* slot_table;  /* [n][num_cols] */
    const int32_t* accepted;    /* [n], values 1 .. num_cols, or NULL */
    const uint8_t* reset;       /* [n] or NULL: nonzero starts request r from a zero state */
    const void* q;              /* [total][h_qk][k], 16-byte aligned */
    const void* k;              /* [total][h_qk][k], 16-byte aligned */
    const void* v;              /* [total][hv][v], 16-byte aligned */
    const float* a;             /* [total][hv][k], 16-byte aligned */
    const float* b;             /* [total][hv] */
    const float* a_log;         /* [hv] or NULL */
    const float* dt_bias;       /* [hv][k] or NULL */
    float* o;                   /* [total][hv][v] (output) */
} kda_step_args;

/*
 * The general step (accepted-length speculative decode, variable-length
 * requests, padding, grouped heads, learned gate scale) on one pool; see
 * kda_step_args.  args is a host pointer.  Host checks (before any launch):
 * KDA_ERR_NULL, _DTYPE_*, _SHAPE (h_qk not dividing hv, num_cols < 1, max_t >
 * num_cols, total inconsistent with n and max_t, in_place with cu_seqlens or
 * max_t != 1), _ALIGN, _ARG (negative counts, reserved != 0, unknown flags).
 * Device checks (in *dev_status, the tile skipped): KDA_ERR_ARG for an
 * accepted column outside 1 .. num_cols or token offsets outside 0 .. max_t;
 * KDA_ERR_SLOT_RANGE for a slot id >= num_slots.  KDA_LAUNCH_PDL_EARLY_STATE
 * also lets the kernel read cu_seqlens, accepted and slot_table early.
 * n == 0 or total == 0 is a no-op after the pool checks.
 */
int kda_step(const kda_pool* pool, const kda_step_args* args, int32_t* dev_status, uint32_t flags,
             void* stream);

/*
 * The causal short convolution in front of the recurrence, with its paged
 * window (pull request 2894, review thread on the conv window: the conv pool
 * keeps kernel - 1 + num_spec inputs per request; a step reads its kernel - 1
 * history entries at the accepted index and writes back the kept old entries
 * followed by its inputs).  One window per slot: [state_len][channels] of
 * `dtype`, oldest entry first, channel innermost:
 *   entry e, channel c of slot s = base + s * slot_stride + e * channels + c.
 */
typedef struct kda_conv_window {
    void* base;           /* device */
    int32_t dtype;        /* KDA_F32, KDA_F16 or KDA_BF16: also the dtype of x and y */
    int32_t channels;     /* C >= 1 */
    int32_t state_len;    /* L: kernel_width - 1 .. 32 */
    int32_t reserved;     /* 0 */
    int64_t num_slots;
    int64_t slot_stride;  /* elements from one slot to the next, >= state_len * channels */
} kda_conv_window;

/*
 * Arguments of kda_conv_step (device pointers unless noted; optional ones may
 * be NULL).  Request r owns tokens cu_seqlens[r] .. cu_seqlens[r+1] - 1 of x
 * and y (or r * max_t .. with cu_seqlens NULL; T_r <= max_t) and the window
 * of slot conv_slot[r] (negative: a padding request, nothing read or stored,
 * its y rows zero).  With acc = accepted[r] - 1 (0 when accepted is NULL),
 * m = acc + kernel_width - 1 and kept = max(0, state_len - T_r):
 *   history h_i = W[acc + i], i < kernel_width - 1 (zeros when reset[r]);
 *   y_t = act(bias + sum_i weight[i] z[t + i]) with z = h ++ x (weight[kernel_width - 1]
 *   weighs x_t); act = SiLU (x sigmoid(x)) when activation == 1, none when 0;
 *   the window becomes W[m - kept .. m - 1] (zeros when reset[r]) followed by
 *   the last min(T_r, state_len) inputs.  T_r == 0 leaves the window alone.
 * Arithmetic is fp32; y is rounded to nearest even; the window keeps exact
 * copies of x.  Device checks (in *dev_status, that request skipped):
 * KDA_ERR_ARG unless 0 <= acc, m <= state_len and kept <= m, and for offsets
 * outside 0 .. max_t; KDA_ERR_SLOT_RANGE for conv_slot[r] >= num_slots.
 */
typedef struct kda_conv_args {
    int32_t n;                  /* requests */
    int32_t total;              /* packed tokens: rows of x and y */
    int32_t max_t;              /* most tokens of any request */
    int32_t kernel_width;       /* 1 .. 8 */
    int32_t activation;         /* 0 none, 1 SiLU */
    int32_t reserved;           /* 0 */
    const int32_t* cu_seqlens;  /* [n + 1] or NULL */
    const int32_t* conv_slot;   /* [n] */
    const int32_t* accepted;    /* [n] or NULL */
    const uint8_t* reset;       /* [n] or NULL */
    const void* x;              /* [total][channels] of the window's dtype */
    const float* weight;        /* [channels][kernel_width] */
    const float* bias;          /* [channels] or NULL */
    void* y;                    /* [total][channels] of the window's dtype (output) */
} kda_conv_args;

/*
 * One step of the short convolution (see kda_conv_args); win and args are host
 * pointers.  Host checks: KDA_ERR_NULL, _DTYPE_UNSUPPORTED (window dtype),
 * _SHAPE (channels < 1, kernel_width outside 1..8, state_len outside
 * kernel_width - 1 .. 32, slot_stride too small, total inconsistent with n and
 * max_t), _ALIGN (x, y, base to their element size; ids, weight, bias 4-byte),
 * _ARG (negative counts, activation not 0/1, reserved fields, unknown flags).
 * Works in either library build (the window dtype is independent of the pool's).
 * n == 0 or total == 0 is a no-op.
 */
int kda_conv_step(const kda_conv_window* win, const kda_conv_args* args, int32_t* dev_status,
                  uint32_t flags, void* stream);

/*
 * Arguments of kda_decode_conv_step: one decode token per request with the
 * short convolution in front of the recurrence done in the same kernel (pull
 * request 2894, review thread on the conv window: the conv runs on the
 * inputs right before the recurrence; pull request 2130, What: the decode
 * step).  x holds each request's pre-convolution inputs of the three streams
 * side by side, channels = 2 * h_qk * k + hv * v (pool's hv, k, v):
 *   q channels  [0, h_qk k)            head g, row i at g k + i
 *   k channels  [h_qk k, 2 h_qk k)     head g, row i at h_qk k + g k + i
 *   v channels  [2 h_qk k, channels)   head h, column j at 2 h_qk k + h v + j
 * Per request r the call is, bit for bit, kda_conv_step with one token
 * (conv_slot[r], no accepted index, the same reset flag) followed by
 * kda_decode_step on slot_ids[r] whose q, k, v are that step's y, read as
 * the window's dtype; value head h reads q/k head h / (hv / h_qk).  The
 * window must hold kernel_width - 1 or kernel_width entries (a one-token step
 * keeps state_len - 1 old ones, which must lie within the history it reads).
 *   slot_ids, conv_slot  device int32 [n]: the state slot and the window slot.
 *   reset     device uint8 [n] or NULL: zero state and zero history.
 *   x         device [n][channels] of the window's dtype.
 *   weight    device fp32 [channels][kernel_width];  bias device fp32 [channels] or NULL.
 *   a, b, o   as for kda_decode_step: fp32 [n][hv][k] (16-byte aligned), [n][hv], [n][hv][v].
 *   y         device [n][channels] of the window's dtype, or NULL: the
 *             convolution's outputs, when the caller wants them as well.
 *   a_log, dt_bias  device fp32 [hv] and [hv][k], or NULL: the layer's learned
 *             gate scale and bias, alpha = exp(-exp(a_log[h]) softplus(a + dt_bias[h])),
 *             as for kda_step (which the call then matches in place of kda_decode_step).
 *   counters  device int32 [n][h_qk], all zero on entry (allocate once and
 *             zero once); the call leaves them zero.  Several CTAs read one
 *             q/k channel's window, so the last of them to finish reading
 *             writes the new entries; each counts its read here.
 */
typedef struct kda_decode_conv_args {
    int32_t n;                  /* requests */
    int32_t h_qk;               /* q/k heads: divides the pool's hv */
    int32_t kernel_width;       /* 1 .. 4 */
    int32_t activation;         /* 0 none, 1 SiLU */
    const int32_t* slot_ids;    /* [n] */
    const int32_t* conv_slot;   /* [n] */
    const uint8_t* reset;       /* [n] or NULL */
    const void* x;              /* [n][channels] */
    const float* weight;        /* [channels][kernel_width] */
    const float* bias;          /* [channels] or NULL */
    const float* a;             /* [n][hv][k] */
    const float* b;             /* [n][hv] */
    float* o;                   /* [n][hv][v] (output) */
    void* y;                    /* [n][channels] (output) or NULL */
    int32_t* counters;          /* [n][h_qk] */
    const float* a_log;         /* [hv] or NULL: the learned gate scale, as in kda_step */
    const float* dt_bias;       /* [hv][k] or NULL: the gate bias, as in kda_step */
} kda_decode_conv_args;

/*
 * One fused conv + decode step (see kda_decode_conv_args); pool, win and args
 * are host pointers.  Host checks: those of kda_decode_step for the pool,
 * KDA_ERR_NULL, _DTYPE_UNSUPPORTED (window dtype), _SHAPE (channels other
 * than 2 h_qk k + hv v, h_qk not dividing hv, kernel_width outside 1 .. 4,
 * state_len outside kernel_width - 1 .. kernel_width, slot_stride too small),
 * _ALIGN (x, y, window base to their element size, a to 16 bytes, the rest to
 * 4), _ARG (negative n, activation not 0/1, flags other than the PDL bits).
 * Device checks (in *dev_status, the request skipped whole, its counters left
 * alone): KDA_ERR_SLOT_RANGE for a slot id or window slot outside the pool.
 * KDA_LAUNCH_PDL_EARLY_STATE lets the kernel read the slot ids, reset flags,
 * state tiles, weights, bias and the window's history entries before the
 * previous kernel has completed (which must then step neither this pool nor
 * this window); x is read, and the window, counters, y and o are written,
 * only after it has completed.  The window is rewritten at the end of each
 * CTA's work, off the recurrence's path.
 * n == 0 is a no-op after the host checks.
 */
int kda_decode_conv_step(const kda_pool* pool, const kda_conv_window* win, const kda_decode_conv_args* args,
                         int32_t* dev_status, uint32_t flags, void* stream);

/*
 * The convolution half of kda_step_conv: the general speculative step with the
 * short convolution done in the same kernel (pull request 2894, review thread
 * on the conv window: the window keeps kernel - 1 + num_spec inputs, a step
 * reads its history at the accepted index and writes back the kept old
 * entries followed by its inputs).  x holds each token's pre-convolution
 * q | k | v inputs, channels = 2 * h_qk * k + hv * v, laid out as for
 * kda_decode_conv_args.  Per call the result is, bit for bit, kda_conv_step
 * over the same requests (cu_seqlens, accepted, reset; conv_slot[r]; a padding
 * request's window left alone and its y rows zero) followed by kda_step with
 * q, k, v taken from that y, read as the window's dtype.
 *   conv_slot  device int32 [n]: the window slot of request r (ignored for a
 *              padding request).
 *   x          device [total][channels] of the window's dtype.
 *   weight     device fp32 [channels][kernel_width];  bias device fp32 [channels] or NULL.
 *   y          device [total][channels] of the window's dtype, or NULL.
 *   counters   device int32 [n][h_qk], zero on entry; the call leaves them zero
 *              (as for kda_decode_conv_args).
 */
typedef struct kda_step_conv_args {
    int32_t kernel_width;       /* 1 .. 4 */
    int32_t activation;         /* 0 none, 1 SiLU */
    const int32_t* conv_slot;   /* [n] */
    const void* x;              /* [total][channels] */
    const float* weight;        /* [channels][kernel_width] */
    const float* bias;          /* [channels] or NULL */
    void* y;                    /* [total][channels] (output) or NULL */
    int32_t* counters;          /* [n][h_qk] */
} kda_step_conv_args;

/*
 * One speculative step with the convolution fused in front (see
 * kda_step_conv_args); pool, step, win and conv are host pointers.  step is as
 * for kda_step with in_place = 0, max_t <= 8 (one chunk of tokens a request),
 * q, k and v NULL (the convolution makes them) and qkv_dtype the window's
 * dtype.  Host checks: those of kda_step, then KDA_ERR_ARG (in_place set, q/k/v
 * given, qkv_dtype not the window's, activation not 0/1, flags other than the
 * PDL bits), KDA_ERR_SHAPE (max_t above 8, channels other than
 * 2 h_qk k + hv v, kernel_width outside 1 .. 4, state_len outside
 * kernel_width - 1 .. 32, slot_stride too small), _ALIGN, _NULL.  Device
 * checks (the request skipped whole, its counters left alone): a window slot
 * outside the pool, KDA_ERR_SLOT_RANGE; acc + kernel_width - 1 > state_len
 * or more kept entries than that (acc = accepted[r] - 1), KDA_ERR_ARG.
 * KDA_LAUNCH_PDL_EARLY_STATE also lets the kernel read the window slots,
 * weights, bias and history entries early; x is read, and the window,
 * counters, y and outputs are written, only after the previous kernel has
 * completed.  n == 0 or total == 0 is a no-op after the host checks.
 */
int kda_step_conv(const kda_pool* pool, const kda_step_args* step, const kda_conv_window* win,
                  const kda_step_conv_args* conv, int32_t* dev_status, uint32_t flags, void* stream);

/*
 * Arguments of kda_prefill: the recurrence over packed prompts (the second
 * workload of pull request 2130, What: prefill reads and writes the state
 * through the destination's element type like every other path).  Request r
 * owns tokens cu_seqlens[r] .. cu_seqlens[r+1] - 1 (or r * max_t .. with
 * cu_seqlens NULL); its state starts from slot init_slot[r] (zero when
 * reset[r] is nonzero: a fresh prompt; a negative init_slot is a padding
 * request, nothing read or stored, outputs zero) and, after its last token,
 * is stored to final_slot[r] (negative: not stored; it may equal init_slot[r]).
 * No per-token state is stored.  A request with no tokens stores its initial
 * state (zero on a reset) to final_slot[r] unchanged: the state after its last
 * token is the one it started from, so a prompt split into an empty part and
 * the rest gives the same final state as the whole prompt.
 * Heads, gate and layouts as in kda_step_args; o gets every token's output.
 */
typedef struct kda_prefill_args {
    int32_t n;                  /* requests */
    int32_t total;              /* packed tokens */
    int32_t max_t;              /* most tokens of any request */
    int32_t h_qk;               /* q/k heads; hv % h_qk == 0 */
    int32_t qkv_dtype;          /* KDA_F32, KDA_F16 or KDA_BF16 */
    int32_t reserved;           /* 0 */
    const int32_t* cu_seqlens;  /* [n + 1] or NULL */
    const int32_t* init_slot;   /* [n] */
    const int32_t* final_slot;  /* [n] */
    const uint8_t* reset;       /* [n] or NULL */
    const void* q;              /* [total][h_qk][k], 16-byte aligned */
    const void* k;              /* [total][h_qk][k], 16-byte aligned */
    const void* v;              /* [total][hv][v], 16-byte aligned */
    const float* a;             /* [total][hv][k], 16-byte aligned */
    const float* b;             /* [total][hv] */
    const float* a_log;         /* [hv] or NULL */
    const float* dt_bias;       /* [hv][k] or NULL */
    float* o;                   /* [total][hv][v] (output) */
} kda_prefill_args;

/*
 * Prefill (see kda_prefill_args).  Host checks as for kda_step (KDA_ERR_SHAPE
 * for total != n * max_t without cu_seqlens); device: KDA_ERR_ARG for offsets
 * outside 0 .. max_t or past total, KDA_ERR_SLOT_RANGE for a slot >= num_slots.
 * n == 0 is a no-op.  total == 0 with n > 0 still stores every request's
 * initial state to its final slot; q, k, v, a, b and o may then be NULL.
 */
int kda_prefill(const kda_pool* pool, const kda_prefill_args* args, int32_t* dev_status, uint32_t flags,
                void* stream);

/*
 * Prefill in two passes over chunks of 16 tokens: a pass over every (chunk,
 * head) at once that depends on the inputs only, then a short sequential scan
 * per (request, head, 32 value columns) that carries the state from chunk to
 * chunk.  Same arguments and results as kda_prefill; the first pass's results
 * go to a caller-provided device workspace of at least
 * kda_prefill_workspace_bytes(...) bytes, 256-byte aligned (KDA_ERR_ARG when
 * smaller, KDA_ERR_ALIGN when misaligned).  K and V at most 128, as everywhere.
 */
int kda_prefill_workspace_bytes(const kda_pool* pool, int32_t n, int32_t total, int64_t* bytes);
int kda_prefill_chunked(const kda_pool* pool, const kda_prefill_args* args, void* workspace,
                        int64_t workspace_bytes, int32_t* dev_status, uint32_t flags, void* stream);

/*
 * kda_prefill_chunked without a caller workspace, allocating nothing, for
 * callers that cannot call cudaMalloc (inside a stream capture whose
 * allocation mode forbids it, or a runtime that hands out no device memory):
 * the first pass's results go to a scratch buffer of KDA_PREFILL_SCRATCH_BYTES
 * that each library build holds in device memory as a file-scope array,
 * resident on every device where the library's module is loaded, for the life
 * of the process.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  KDA_ERR_SHAPE when kda_prefill_workspace_bytes(...) exceeds the
 * buffer (at HV=12, K=V=128 it holds about 4K tokens).  Every call shares the
 * buffer, and calls that overlap on the GPU race on it: order them (one
 * stream, or streams synchronised between calls).  The pages have no
 * counterpart; otherwise as kda_prefill_chunked.
 */
#define KDA_PREFILL_SCRATCH_BYTES (128ll << 20)
int kda_prefill_chunked_noalloc(const kda_pool* pool, const kda_prefill_args* args, int32_t* dev_status,
                                uint32_t flags, void* stream);

/*
 * Staging of a step's inputs from host memory by a kernel.  copies[i] moves
 * `bytes` bytes from `src`, pinned host memory mapped into the device's address
 * space (cudaHostAlloc / cudaMallocHost memory; pageable memory is refused),
 * to `dst`, device memory; both 16-byte aligned, bytes a multiple of 16.
 * One thread per 16 bytes loads over the host link and stores to the device
 * buffer, all copies in one launch: small per-step transfers then run on the
 * SMs beside other kernels instead of paying the copy engine's fixed cost
 * each.  With KDA_LAUNCH_PDL the loads start before the previous kernel on the
 * stream completes and the stores wait for it.  copies: host array of
 * n <= KDA_STAGE_MAX_COPIES entries.  Host checks: KDA_ERR_ARG (n out of
 * range, bytes negative or not a multiple of 16, a source that is not
 * device-mapped host memory or a destination that is not device memory,
 * flags other than KDA_LAUNCH_PDL), KDA_ERR_NULL, KDA_ERR_ALIGN.  The pages
 * have no counterpart: this serves the end-to-end measurement of a step fed
 * from host buffers.
 */
#define KDA_STAGE_MAX_COPIES 8
typedef struct kda_host_copy {
    void* dst;          /* device */
    const void* src;    /* pinned, device-mapped host memory */
    int64_t bytes;
} kda_host_copy;
int kda_stage_host(const kda_host_copy* copies, int32_t n, uint32_t flags, void* stream);

/*
 * Checkpoint planes (ReplaySSM in pull request 2945, Changes: the checkpoint
 * load and the flush go through state_at; pull request 2130, What: the plane
 * shapes and the checkpoint layout id derive from the state dtype, so a build
 * that flips the dtype cannot read another's checkpoint images).
 *
 * kda_layout_id: the layout id of `pool`'s states, a 32-bit FNV-1a digest of
 * the five int32 values (1, dtype, hv, k, v); two pools share it exactly when
 * their states are interchangeable byte for byte.  0 for a NULL pool.
 */
uint32_t kda_layout_id(const kda_pool* pool);

/*
 * A plane of checkpoint entries, each one slot's state in the pool's layout:
 * entry e = base + e * entry_stride elements.  layout_id is the
 * kda_layout_id of the pool the plane serves (it travels with the image).
 */
typedef struct kda_ckpt_plane {
    void* base;            /* device, 16-byte aligned */
    uint32_t layout_id;
    int32_t reserved;      /* 0 */
    int64_t num_entries;
    int64_t entry_stride;  /* elements, >= hv * k * v, a multiple of 16 bytes */
} kda_ckpt_plane;

/*
 * kda_ckpt_flush: plane entry entries[i] <- pool slot slots[i];
 * kda_ckpt_load:  pool slot slots[i] <- plane entry entries[i]; i < n.
 * Whole states, bit for bit (no conversion).  A negative slot or entry skips
 * that pair; one past its buffer sets KDA_ERR_SLOT_RANGE in *dev_status and
 * skips it.  Host checks: KDA_ERR_NULL, the pool checks of kda_decode_step,
 * KDA_ERR_LAYOUT when plane->layout_id != kda_layout_id(pool), KDA_ERR_SHAPE
 * for a short entry_stride, KDA_ERR_ALIGN, KDA_ERR_ARG (n < 0, reserved,
 * flags).  slots and entries: device int32 [n].  n == 0 is a no-op.
 */
int kda_ckpt_flush(const kda_pool* pool, const kda_ckpt_plane* plane, const int32_t* slots,
                   const int32_t* entries, int32_t n, int32_t* dev_status, uint32_t flags, void* stream);
int kda_ckpt_load(const kda_pool* pool, const kda_ckpt_plane* plane, const int32_t* slots,
                  const int32_t* entries, int32_t n, int32_t* dev_status, uint32_t flags, void* stream);

/* A static, human-readable string for a kda_status code. */
const char* kda_strerror(int32_t code);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
