/*
 * dmuon.h -- C ABI of the owner-side Muon / AdamW optimizer step on one GPU.
 *
 * The operation: a parameter's single owner updates its own full copy with no
 * communication -- momentum, Newton-Schulz orthogonalisation, weight decay
 * and the parameter update (DMuon docs, "架构设计" (architecture design),
 * §2 "专属归属权——原语", optimizer-step bullet, and §3.3 "Owner 步进";
 * "HSDP 训练（多机）", "底层发生了什么" step 3).  The Newton-Schulz iteration is
 * the one of "架构设计" §1 (X <- aX + bXX^T X + cX(X^T X)^2), applied to the
 * last two dimensions of tensors of rank >= 2 (MindSpore hyper-parallel
 * "分布式 Muon 优化器 — 参数分组设计文档（v2）" §2.1-§2.2).  Non-matrix
 * parameters take the element-wise AdamW routes ("Pure DMuon 路由", route
 * table).  Work units are balanced by the LPT greedy of "架构设计" §3.1.
 *
 * Conventions shared by every entry point:
 *  - Plain pointers and sizes only.  "Device pointer" means memory the
 *    current CUDA device can address (cudaMalloc, or a torch CUDA tensor's
 *    data pointer); "host pointer" means ordinary process memory.
 *  - The caller owns every tensor.  The library owns only what a context
 *    allocates for itself (Newton-Schulz workspace, plan tables), which it
 *    frees in dmuon_context_destroy.
 *  - Device work is enqueued on the caller's stream (a cudaStream_t passed
 *    as void*, NULL = the legacy default stream) and returns without waiting.
 *    Where an entry also uses streams the context owns (the host-buffer
 *    step's copies, the optional momentum overlap), that work starts after
 *    the work already on the caller's stream, and work enqueued there later
 *    runs after it.
 *  - All arguments are validated on the host before anything is enqueued:
 *    a call that returns an error has changed no tensor.
 *  - Results are deterministic: the same inputs give bit-identical outputs
 *    (no floating-point atomics; reductions run in a fixed order).
 *  - Errors are returned as dmuon_status codes; dmuon_last_error() gives a
 *    one-line message for the calling thread's last failure.
 */
#ifndef DMUON_H
#define DMUON_H

#include <stdint.h>

#if defined(__GNUC__)
#define DMUON_API __attribute__((visibility("default")))
#else
#define DMUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dmuon_status {
  DMUON_OK = 0,
  DMUON_ERR_INVALID_ARG = 1, /* null pointer, bad count, bad hyper-parameter      */
  DMUON_ERR_RANK_LT2 = 2,    /* a Muon tensor of rank < 2 (route it to AdamW)     */
  DMUON_ERR_SHAPE = 3,       /* zero or negative dimension, or rank > 4           */
  DMUON_ERR_DTYPE = 4,       /* unsupported gradient dtype                        */
  DMUON_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed                 */
  DMUON_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out (see below)    */
  DMUON_ERR_NOMEM = 7,       /* device or pinned host allocation failed           */
  DMUON_ERR_UNSUPPORTED = 8  /* no usable device (e.g. not sm_100-family)         */
} dmuon_status;

/* Gradient dtypes. */
enum { DMUON_DTYPE_F32 = 0, DMUON_DTYPE_BF16 = 1 };

/* dmuon_muon_step flags. */
enum {
  DMUON_FLAG_NESTEROV = 1u, /* u = g + mu*buf (else u = buf)                      */
  DMUON_FLAG_FP32_NS = 2u   /* validation mode: fp32 Newton-Schulz on CUDA cores  */
};

/* One-line description of a status code.  Never NULL. */
DMUON_API const char* dmuon_status_string(int status);

/* Message of the calling thread's last failed call ("" if none).  Never NULL. */
DMUON_API const char* dmuon_last_error(void);

/*
 * dmuon_lpt_assign -- longest-processing-time greedy assignment.
 *
 * "架构设计" §3.1 "分区（全局 LPT）": one global greedy pass over all work
 * units; on identical slots its makespan is at most 4/3 - 1/(3R) times the
 * optimum.  Tie rules (the page gives none): items in descending size, equal
 * sizes by ascending index; each item to the slot with the smallest load,
 * equal loads to the lowest slot index.  The result is therefore unique.
 *
 *   sizes     host, n_items int64 costs, each >= 0 (read only)
 *   n_items   >= 0
 *   n_slots   >= 1
 *   out_slot  host, n_items int32: slot of each item (written)
 *   out_load  host, n_slots int64: total cost per slot (written), or NULL
 *
 * Pure host code; no CUDA call.  Errors: DMUON_ERR_INVALID_ARG for a null
 * required pointer, n_items < 0, n_slots < 1, a negative size, or a slot
 * load that would overflow int64.
 */
DMUON_API int dmuon_lpt_assign(const int64_t* sizes, int32_t n_items, int32_t n_slots,
                     int32_t* out_slot, int64_t* out_load);

/*
 * dmuon_lpt_assign_layered -- LPT with the two constraints of "架构设计" §3.1
 * ("算法内置的关键约束"): (1) same-layer concurrency: the items of one layer
 * go to different slots, so each owner's broadcast of that layer can run at
 * the same time; (2) small-parameter merging: within a layer, the items
 * below `small_threshold` elements (the page's SMALL_PARAM_THRESHOLD, 5e6 by
 * default) form one unit with one owner.  Units are placed in descending
 * size (ties: lowest first item), each on the least-loaded slot that does
 * not yet hold its layer (ties: lowest index), or on the least-loaded slot
 * overall once every slot holds it.  layers[i] < 0: item i belongs to no
 * layer (never merged, never constrained); with all layers < 0 the result
 * equals dmuon_lpt_assign.
 *
 *   sizes, layers  host, n_items each (read only)
 *   out_slot       host, n_items (written); out_load host, n_slots or NULL
 * Pure host code.  Errors: DMUON_ERR_INVALID_ARG as dmuon_lpt_assign.
 */
DMUON_API int dmuon_lpt_assign_layered(const int64_t* sizes, const int32_t* layers, int32_t n_items,
                                       int32_t n_slots, int64_t small_threshold, int32_t* out_slot,
                                       int64_t* out_load);

/*
 * One Muon-route tensor.  shape[0..rank-1] is row-major and contiguous; the
 * Newton-Schulz iteration acts on the last two dimensions (m rows, n cols)
 * and every leading index is a separate matrix.  All pointers point to
 * rank-shaped contiguous arrays the context's device can dereference:
 *   master      fp32, read and written (the fp32 master weight W)
 *   momentum    fp32, read and written (the momentum buffer)
 *   grad        fp32 or bf16 per grad_dtype, read only
 *   param_bf16  bf16 (raw uint16 bits), written, may be NULL (no bf16 copy)
 * master, momentum and param_bf16 must not overlap one another, any grad, or
 * any written buffer of another tensor of the same call (grads may share
 * memory).  Every entry point checks this on the host, before any launch,
 * and fails with DMUON_ERR_INVALID_ARG naming the two ranges.
 * Tensors whose rows are a multiple of 16 bytes (n % 4 == 0, and n % 8 == 0
 * when param_bf16 is given) with 16-byte-aligned master and param_bf16
 * let the step apply the update inside its last Newton-Schulz product (TMA
 * tile copies from and to those buffers); a call with any other bf16-path
 * tensor applies it in a separate pass for all its tensors, which rounds the
 * last iterate to bf16 first (results stay within the same tolerances).
 * The choice is made over the whole call, so splitting a call into groups
 * (tuning keys 9 and 11, dmuon_step_host) never changes a result.
 * Reachable means memory of the context's device, managed memory, or
 * page-locked host memory mapped into the device's address space
 * (cudaHostAlloc / cudaHostRegister with mapping): the kernels then read
 * grad and write param_bf16 in host memory directly (over NVLink-C2C on a
 * Grace host), with no staging copy.  The step checks every pointer the
 * first time it sees a descriptor array and fails with DMUON_ERR_INVALID_ARG
 * for pageable host memory or another device's memory.
 */
typedef struct dmuon_matrix {
  int32_t rank;          /* 2..4 */
  int32_t grad_dtype;    /* DMUON_DTYPE_F32 or DMUON_DTYPE_BF16 */
  int64_t shape[4];
  float* master;
  float* momentum;
  const void* grad;
  uint16_t* param_bf16;
} dmuon_matrix;

/* One AdamW-route tensor, flattened: numel contiguous elements, every
 * pointer reachable from the context's device in the sense given for
 * dmuon_matrix (checked the same way).  master/exp_avg/exp_avg_sq fp32
 * read+write, grad read only, param_bf16 written (may be NULL).  The
 * written buffers follow dmuon_matrix's no-overlap rule (also across the
 * Muon and AdamW lists of one dmuon_step_host call). */
typedef struct dmuon_vector {
  int64_t numel;
  int32_t grad_dtype;    /* DMUON_DTYPE_F32 or DMUON_DTYPE_BF16 */
  int32_t reserved;
  float* master;
  float* exp_avg;
  float* exp_avg_sq;
  const void* grad;
  uint16_t* param_bf16;
} dmuon_vector;

typedef struct dmuon_context dmuon_context;

/*
 * dmuon_context_create -- a context bound to one CUDA device.
 *   out     host, receives the new context
 *   device  CUDA device ordinal (>= 0)
 * Makes no allocation on the device; workspace is sized on first use and
 * grows as needed.  Errors: DMUON_ERR_INVALID_ARG (null out, device < 0),
 * DMUON_ERR_NOMEM (host allocation).
 */
DMUON_API int dmuon_context_create(dmuon_context** out, int32_t device);

/* Frees every allocation of the context after waiting for its device work.
 * NULL is accepted and ignored. */
DMUON_API int dmuon_context_destroy(dmuon_context* ctx);

/*
 * dmuon_muon_step -- one owner-side Muon step over n tensors.
 *
 * For every 2-D slice (m x n) of every tensor, in fp32 unless noted:
 *   buf <- mu*buf + g;  u <- g + mu*buf (NESTEROV) or u <- buf
 *   X   <- u / (||u||_F + 1e-7), held as X (m <= n) or X^T (m > n) so that
 *          the Gram matrix is p x p with p = min(m, n)
 *   ns_steps times:  A = X X^T;  B = b*A + c*A*A;  X <- a*X + B X
 *          (bf16 operands, fp32 accumulation; fp32 throughout with
 *           DMUON_FLAG_FP32_NS)
 *   W   <- W*(1 - lr*wd) - lr*sqrt(max(1, m/n))*X (in the original
 *          orientation);  param_bf16 <- round-to-nearest-even(W)
 *
 *   ctx       from dmuon_context_create
 *   mats      host array of n descriptors (read during the call only)
 *   n         >= 0 (0 is a no-op)
 *   lr, momentum, wd   finite; ns_steps in [0, 100]; a, b, c finite
 *   flags     DMUON_FLAG_* bits
 *   stream    cudaStream_t of the caller (void*)
 *
 * Errors: DMUON_ERR_INVALID_ARG, DMUON_ERR_RANK_LT2 (rank < 2),
 * DMUON_ERR_SHAPE (rank > 4 or a dimension < 1), DMUON_ERR_DTYPE,
 * DMUON_ERR_NOMEM (workspace), DMUON_ERR_CUDA, DMUON_ERR_UNSUPPORTED.
 * Device-side waits inside the kernels are bounded; if one runs out the
 * kernel records it and returns, and the next dmuon_sync() reports
 * DMUON_ERR_TIMEOUT.  Muon steps on one context must not overlap on the
 * GPU (they share the context's workspace); an AdamW step of the same
 * context may run concurrently on another stream.
 * A call whose tensor list, pointers and settings are unchanged since the
 * previous call on the context enqueues kernel launches only (plan, tables
 * and tensor maps are reused), so it can be captured into a CUDA graph and
 * replayed; the graph fixes the hyper-parameters it was captured with.  The
 * same holds for dmuon_adamw_step (whose step counter is then fixed too).
 */
DMUON_API int dmuon_muon_step(dmuon_context* ctx, const dmuon_matrix* mats, int32_t n,
                    float lr, float momentum, float wd, int32_t ns_steps,
                    float a, float b, float c, uint32_t flags, void* stream);

/*
 * dmuon_muon_step_noalloc -- the Muon step of one tensor, allocating nothing.
 *
 * The pages have no counterpart: this entry exists for callers that cannot
 * call cudaMalloc -- code inside a framework that owns every device
 * allocation through its own pool, code that must not grow its memory after
 * start-up, or code that must not risk the implicit device synchronisation
 * of cudaMalloc/cudaFree.  It computes what dmuon_muon_step computes for
 * `mat`, within the same tolerances and with the same precision policy
 * (bf16 tensor cores for slices with min(m, n) >= 64; the fp32 CUDA-core
 * kernel for min(m, n) < 64 or with DMUON_FLAG_FP32_NS), on the one-CTA
 * tensor-core kernel and with the update in a separate pass (so its bits
 * can differ from dmuon_muon_step's), but needs no context: all scratch
 * (Newton-Schulz buffers, norm partials, descriptor tables, tensor maps,
 * the device error word) lives in one static device array of 64 MiB that
 * every GPU loading this library holds until the process exits, and the
 * host tables are built in a static 1 MiB host buffer.  No cudaMalloc,
 * cudaFree or other allocating routine is called.
 *
 *   mat      host pointer to one descriptor (rank 2..4; leading dims are
 *            separate matrices), device tensors as for dmuon_muon_step
 *   flags    DMUON_FLAG_NESTEROV and/or DMUON_FLAG_FP32_NS
 *   others   as for dmuon_muon_step; stream = cudaStream_t of the caller
 *
 * Works on the current device.  Limits: the tensor's scratch must fit in
 * 64 MiB -- on the bf16 path about 6 bytes per element of every m x n slice
 * plus 6 bytes per element of every p x p Gram (p = min(m, n)), e.g. one
 * 2048 x 2048 matrix; on the fp32 path 8 and 8 -- and its tables in 1 MiB,
 * else DMUON_ERR_SHAPE with the byte counts in dmuon_last_error().  The
 * shape checks of dmuon_muon_step apply as well.
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (once per device, with that device current); make
 * that first call before any stream capture.  Every call shares the one
 * array and it keeps the previous call's contents: calls whose work
 * overlaps on the GPU (different streams, or different host threads without
 * ordering) race on it.
 * Device-side waits are bounded; one that runs out records its site in the
 * array's error word and its kernel returns.  The word is not cleared by a
 * step: dmuon_muon_step_noalloc_sync reports and clears it.
 * Errors: as dmuon_muon_step, plus DMUON_ERR_SHAPE for the size limit.
 */
DMUON_API int dmuon_muon_step_noalloc(const dmuon_matrix* mat, float lr, float momentum, float wd,
                                      int32_t ns_steps, float a, float b, float c, uint32_t flags,
                                      void* stream);

/*
 * dmuon_muon_step_noalloc_sync -- wait for `stream`, then read and clear the
 * error word of dmuon_muon_step_noalloc on the current device (a synchronous
 * copy from the static array; nothing is allocated).  Returns
 * DMUON_ERR_TIMEOUT if a bounded wait ran out since the last such read,
 * DMUON_ERR_CUDA if the stream reported an error, else DMUON_OK.
 */
DMUON_API int dmuon_muon_step_noalloc_sync(void* stream);

/*
 * dmuon_adamw_step -- one AdamW step over n flattened tensors ("Pure DMuon
 * 路由": routes "adamw" and "sharded_adamw" both run AdamW; the shard
 * placement is outside this call).  In fp32, per element:
 *   m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2
 *   W <- W*(1 - lr*wd) - (lr/(1-b1^t)) * m / (sqrt(v)/sqrt(1-b2^t) + eps)
 *   param_bf16 <- round-to-nearest-even(W)
 *   step = t >= 1.  beta1, beta2 in [0, 1); eps >= 0; lr, wd finite.
 * Errors as dmuon_muon_step.
 */
DMUON_API int dmuon_adamw_step(dmuon_context* ctx, const dmuon_vector* ts, int32_t n,
                     float lr, float beta1, float beta2, float eps, float wd,
                     int64_t step, void* stream);

/* Host side of one tensor in dmuon_step_host: page-locked host buffers
 * (cudaHostAlloc, or cudaHostRegister'ed) with the tensor's shape.
 *   grad_host   this step's gradient, dtype = the descriptor's grad_dtype;
 *               read (copied into the descriptor's device grad buffer)
 *   param_host  bf16 parameter; written (copied from the descriptor's device
 *               param_bf16 buffer, which must then be non-NULL); NULL = the
 *               parameter stays on the device only */
typedef struct dmuon_host_io {
  const void* grad_host;
  uint16_t* param_host;
} dmuon_host_io;

/* Hyper-parameters of dmuon_step_host, as the scalar arguments of
 * dmuon_muon_step and dmuon_adamw_step. */
typedef struct dmuon_muon_hparams {
  float lr, momentum, wd;
  int32_t ns_steps;
  float a, b, c;
  uint32_t flags;
} dmuon_muon_hparams;

typedef struct dmuon_adamw_hparams {
  float lr, beta1, beta2, eps, wd;
  int32_t reserved;  /* 0 */
  int64_t step;
} dmuon_adamw_hparams;

/*
 * dmuon_step_host -- one owner step whose gradients arrive in host memory and
 * whose bf16 parameters go back to host memory.
 *
 * The pages have no counterpart: their owner step ("架构设计" §3.3 "Owner
 * 步进") starts from gradients already in the owner's device memory.  This
 * entry serves callers whose gradients and parameters live in host memory,
 * and adds only the copies around the same computation.  For every tensor
 * it copies io.grad_host into the descriptor's device grad buffer, runs
 * exactly dmuon_muon_step (mats, *muon) and dmuon_adamw_step (vecs,
 * *adamw), and copies the device param_bf16 buffer into io.param_host.  The
 * Muon tensors are cut into up to n_groups consecutive groups of about equal
 * Newton-Schulz work (1 <= n_groups <= 64; fewer for short lists, since
 * every group holds at least 2^25 elements, dmuon_set_tuning key 11); each
 * group's gradients travel while earlier groups compute and each group's parameters
 * travel while later groups compute, on two copy streams the context owns,
 * so the host link is busy only at the ends of the step.  The AdamW tensors
 * travel and step right after the first Muon group.  Parameter copies start
 * once every gradient copy has landed (where the link's two directions
 * share a bottleneck, earlier ones would slow the gradient copies the
 * compute waits for).  Results are bit-identical
 * to the device entry points on the same inputs.
 *
 *   mats, mat_io  n_mats Muon tensors and their host buffers
 *   muon          Muon hyper-parameters (non-NULL if n_mats > 0)
 *   vecs, vec_io  n_vecs AdamW tensors and their host buffers
 *   adamw         AdamW hyper-parameters (non-NULL if n_vecs > 0)
 *   stream        all work is ordered after the work already on `stream`,
 *                 and work enqueued on `stream` later runs after the last
 *                 parameter copy has landed in host memory
 * Host buffers are checked once per descriptor array: pageable host memory
 * is refused (DMUON_ERR_INVALID_ARG).  Other errors as dmuon_muon_step and
 * dmuon_adamw_step.  Shares the context's workspace with dmuon_muon_step:
 * the two must not overlap on the GPU.
 */
DMUON_API int dmuon_step_host(dmuon_context* ctx,
                              const dmuon_matrix* mats, const dmuon_host_io* mat_io, int32_t n_mats,
                              const dmuon_muon_hparams* muon,
                              const dmuon_vector* vecs, const dmuon_host_io* vec_io, int32_t n_vecs,
                              const dmuon_adamw_hparams* adamw,
                              int32_t n_groups, void* stream);

/*
 * dmuon_sync -- wait for the stream and report device-side errors.
 * Synchronises `stream`, then reads and clears the context's device error
 * word.  Returns DMUON_ERR_TIMEOUT if a bounded wait ran out since the last
 * call, DMUON_ERR_CUDA if the stream reported an error, else DMUON_OK.
 */
DMUON_API int dmuon_sync(dmuon_context* ctx, void* stream);

/*
 * dmuon_selftest_wait_timeout -- exercise the bounded-wait failure path.
 * Launches one block that waits on a barrier nothing will complete, giving
 * up after timeout_us microseconds (1..2,000,000); the kernel records the
 * timeout and returns normally, leaving the context usable.  A following
 * dmuon_sync() returns DMUON_ERR_TIMEOUT.  With ctx == NULL the timeout is
 * recorded in the error word of dmuon_muon_step_noalloc on the current
 * device instead, and dmuon_muon_step_noalloc_sync() reports it.  Used by
 * the failure-detection tests; never part of an optimizer step.
 */
DMUON_API int dmuon_selftest_wait_timeout(dmuon_context* ctx, int32_t timeout_us, void* stream);

/*
 * dmuon_set_tuning -- process-wide defaults of the kernel and planning
 * policy.  Every context copies them when it is created
 * (dmuon_context_create); contexts that exist already keep their own copy,
 * which dmuon_context_set_tuning changes.  Keys and values:
 *   key 2: tensor-core kernel of the Newton-Schulz phases (1 = CTA pairs,
 *          cta_group::2, on 256 x 256 tiles and, per key 12, 256 x 512
 *          ones, the default; 0 = one CTA per 128 x 256 tile).
 *   key 3: pipeline depth of the CTA-pair kernel (4 or 5 stages; default 4;
 *          the last Combine with the fused update always runs 4).
 *   key 4: tile order inside a problem (1 = longer tile dimension outer, the
 *          default; 0 = rows outer).  Takes effect at the next plan build.
 *   key 6: CTA-pair kernel keeps symmetric products as upper blocks only and
 *          reads them through transposed loads (1) or stores mirrored copies
 *          of off-diagonal blocks (0).
 *   key 7: from the third Newton-Schulz iteration on, the a*X term is folded
 *          into the polynomial matrix, X' = (a I + B) X, so the last product
 *          reads no extra operand (1, default), or added in the epilogue (0).
 *   key 8: CTA-pair kernel: a launch whose tiles average fewer than `value`
 *          64-deep k-blocks drains its accumulators with 8 epilogue warps
 *          instead of 4 (default 32; 0 = always 4, a large value = always 8
 *          except for the fused update).
 *   key 9: a Muon step is cut into up to `value` groups of consecutive
 *          tensors (1..16, default 1), each of at least key 10's size;
 *          group g+1's momentum pass runs on a side stream of the context
 *          while group g's Newton-Schulz products run on the caller's
 *          stream.  1 = all on the caller's stream.  Results do not depend
 *          on the setting.
 *   key 10: smallest group of key 9, in units of 2^20 elements (1..65536,
 *          default 1024).
 *   key 11: smallest group of dmuon_step_host, in units of 2^10 elements
 *          (1..2^20, default 32768).
 *   key 12: CTA-pair kernel: a launch (other than a fused update) whose
 *          tiles average at least `value` 64-deep k-blocks runs 256 x 512
 *          tiles wherever two adjacent column blocks exist (0..1e6, default
 *          128; 0 = never).  Results do not depend on the setting.
 * Results never depend on keys 3, 4, 6, 8, 9, 10, 11 and 12 (bit for bit);
 * key 2 changes the kernel and key 7 the rounding points, both within the
 * documented tolerances.
 * Returns DMUON_ERR_INVALID_ARG for an unknown key or a value out of range
 * (nothing changes then).  Thread-safe (the defaults are guarded by a lock).
 */
DMUON_API int dmuon_set_tuning(int32_t key, int32_t value);

/*
 * dmuon_context_set_tuning -- the same keys and values as dmuon_set_tuning,
 * for one context only (its copy of the defaults).  Takes effect at the
 * context's next step.  Must not be called while another thread uses the
 * context.  Errors: DMUON_ERR_INVALID_ARG for a null context, an unknown
 * key or a value out of range (nothing changes then).
 */
DMUON_API int dmuon_context_set_tuning(dmuon_context* ctx, int32_t key, int32_t value);

/* Kernel kinds reported by dmuon_profile_read. */
enum {
  DMUON_KERNEL_MOMENTUM = 0, /* momentum + X0 + sum of squares      */
  DMUON_KERNEL_NORM = 1,     /* per-slice 1/(||u|| + eps)            */
  DMUON_KERNEL_NS_GRAM = 2,  /* A = X X^T (or X^T X)                 */
  DMUON_KERNEL_NS_POLY = 3,  /* B = b A + c A A                      */
  DMUON_KERNEL_NS_COMBINE = 4, /* X <- a X + B X (or a X + X B)      */
  DMUON_KERNEL_UPDATE = 5,   /* weight decay + update + bf16 copy    */
  DMUON_KERNEL_ADAMW = 6,
  DMUON_KERNEL_KINDS = 7
};

/*
 * dmuon_profile -- per-kernel device timing (tracing).
 * With enable != 0 every later launch of the context is bracketed by two
 * CUDA events recorded on the launching stream; with enable == 0 no events
 * are recorded.  Errors: DMUON_ERR_INVALID_ARG for a null context.
 */
DMUON_API int dmuon_profile(dmuon_context* ctx, int32_t enable);

/*
 * dmuon_profile_read -- totals since the previous read, then reset.
 *   ms_out     host, DMUON_KERNEL_KINDS doubles: summed device milliseconds
 *   count_out  host, DMUON_KERNEL_KINDS int64: launches (may be NULL)
 * Waits for the recorded events (host blocks until those launches finish).
 * Errors: DMUON_ERR_INVALID_ARG (null ctx or ms_out), DMUON_ERR_CUDA.
 */
DMUON_API int dmuon_profile_read(dmuon_context* ctx, double* ms_out, int64_t* count_out);

/*
 * dmuon_profile_host_timeline -- where the time of a host-buffer step went.
 * For the last dmuon_step_host call made on the context while profiling was
 * enabled (dmuon_profile), waits for its events and writes, in
 * milliseconds since the call's work started on its stream:
 *   ms_out[0]            all gradient copies (host to device) done
 *   ms_out[1]            all copies done (the step's end)
 *   ms_out[2 + 3g + 0]   group g's gradient copies done
 *   ms_out[2 + 3g + 1]   group g's compute done
 *   ms_out[2 + 3g + 2]   group g's parameter copies (device to host) done
 * for the call's G groups (*n_groups_out = G; 0 and nothing written if no
 * such call was recorded).  capacity = doubles available in ms_out; fewer
 * than 2 + 3G gives DMUON_ERR_INVALID_ARG (with *n_groups_out set).
 */
DMUON_API int dmuon_profile_host_timeline(dmuon_context* ctx, double* ms_out, int32_t capacity,
                                          int32_t* n_groups_out);

/*
 * dmuon_kernel_launches -- number of kernels the context has launched since
 * it was created (host-side count, for benchmarking).  Returns -1 for NULL.
 */
DMUON_API int64_t dmuon_kernel_launches(const dmuon_context* ctx);

#ifdef __cplusplus
}
#endif

#endif /* DMUON_H */
