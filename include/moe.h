/*
 * int4_routed_expert_moe_gb300 -- C ABI of the routed INT4-expert MoE FFN
 * for NVIDIA GB300 (sm_103a), one process on one GPU.
 *
 * What the library computes (sources are web pages, cited by title/section):
 *   * "Horizon RunMap -- Prévia Técnica", "02 / A solução" and
 *     "03 / Arquitetura": the router chooses the experts of each token; the
 *     expert kernel combines compact expert weights and FP16 scales with FP16
 *     activations and returns the result to the rest of the model, without
 *     keeping an expanded expert on the GPU. The non-routed parts run in FP16.
 *   * same page, "08 / Comportamento do modelo": W4A16 -- routed expert
 *     weights INT4 with FP16 scales, FP16 activations, conversion inside the
 *     kernel, FP32 accumulation with explicit rounding points.
 *   * same page, "03 / Arquitetura", contract resident-qpacked-cache-v1
 *     (ADR 0009): complete immutable source in host RAM, copies arrive at a
 *     GPU position and are published as a whole new generation, an evicted
 *     copy is reused only after its readers retire, capacity is fixed before
 *     requests and init rejects a profile that is short of it, a failure
 *     before publish keeps the previous generation.
 *   * "Desenvolvedor do Strata cria mapa ao vivo de 24 576 especialistas MoE
 *     em uma GTX 1070": hot experts stay in VRAM; eviction follows an access
 *     counter whose old accesses lose weight.
 *   * lucashiago.com.br "local" explainer, etapa 1: every block of weights
 *     carries a scale and a zero point that rebuild it.
 *
 * Conventions for every call:
 *   * Pointers documented "device" must point to GPU memory of the current
 *     device; "host" pointers to CPU memory. The caller owns every buffer
 *     passed in (allocate with any allocator); the library owns only the
 *     residency handle and the CUDA events inside it.
 *   * `stream` is a cudaStream_t (NULL = legacy default stream). GPU calls
 *     only enqueue work on it and return; nothing synchronises the device
 *     unless stated.
 *   * Every call returns a moe_status (0 = MOE_OK). No call aborts, throws
 *     or traps. moe_last_error() gives a thread-local detail string for the
 *     last failure. An asynchronous CUDA error from earlier work is reported
 *     by the next call that checks (MOE_ERR_CUDA).
 *   * FP16 values are passed as their 16-bit patterns (IEEE binary16).
 *
 * Expert block (one expert, `moe_expert_block_bytes` bytes; H = hidden,
 * I = inter, g = group). Two sections of fixed-stride rows, so that the rows
 * a kernel needs of one expert are one contiguous byte range:
 *   gate/up section: I rows n, stride gu_row_bytes, each holding
 *     [codes of W_g row n: H/2 bytes][codes of W_u row n: H/2 bytes]
 *     [H/g quads of fp16 (s_gate, z_gate, s_up, z_up), one per group]
 *   down section (at d_offset = I * gu_row_bytes): H rows m, stride
 *     d_row_bytes, each holding
 *     [codes of W_d row m: I/2 bytes][I/g pairs of fp16 (s_down, z_down)]
 * Strides are the row contents rounded up to 16 bytes (moe_expert_block_layout
 * gives every offset). Byte c of a code row holds element 2c in its low
 * nibble and element 2c+1 in its high nibble; codes are unsigned 0..15. The
 * weight is
 *   W[n][c] = (q[n][c] - z[n][c/g]) * s[n][c/g],
 * groups running along each row's reduction axis (H for gate/up, I for down).
 * Without padding (H/g and I/g even) a block holds 3*H*I/2 + 3*(H*I/g)*4
 * bytes, which is also the byte count every read of one expert moves.
 * Shape limits: H and I multiples of 64, g a multiple of 32 dividing H and I,
 * H <= 8192, I <= 8192.
 */
#ifndef INT4_ROUTED_EXPERT_MOE_GB300_MOE_H
#define INT4_ROUTED_EXPERT_MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,         /* null pointer, bad enum, k > E, ...            */
  MOE_ERR_SHAPE = -2,       /* shape outside the limits above                */
  MOE_ERR_CAPACITY = -3,    /* residency capacity or workspace too small     */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime call failed                    */
  MOE_ERR_NONFINITE = -5,   /* NaN / +inf router logits (host-side checks)   */
  MOE_ERR_STATE = -6,       /* handle used in a state that forbids the call  */
  MOE_ERR_TIMEOUT = -7,     /* a bounded device wait gave up                 */
  MOE_ERR_INJECTED = -8,    /* failure injected by the residency test hook   */
  MOE_ERR_UNSUPPORTED = -9  /* valid request this build does not implement   */
} moe_status;

typedef struct {
  int32_t hidden; /* H */
  int32_t inter;  /* I, the expert intermediate size */
  int32_t group;  /* g, elements per scale/zero group */
} moe_expert_shape;

/* ---- diagnostics --------------------------------------------------------- */
const char* moe_status_string(int status);
/* Thread-local detail of the last failing call on this thread ("" if none). */
const char* moe_last_error(void);
/* Library ABI version, currently 1. */
int moe_version(void);

/* ---- expert block layout (host only) ------------------------------------- */
typedef struct {
  uint64_t total;        /* bytes of one expert block */
  uint64_t d_offset;     /* byte offset of the down section (I * gu_row_bytes) */
  uint32_t gu_row_bytes; /* stride of the I gate/up rows (multiple of 16) */
  uint32_t d_row_bytes;  /* stride of the H down rows (multiple of 16) */
  /* byte offsets inside a gate/up row: codes, then the scale/zero quads */
  uint32_t gu_q_gate, gu_q_up, gu_sz;
  /* byte offsets inside a down row: codes, then the scale/zero pairs */
  uint32_t d_q, d_sz;
} moe_block_layout;

/* Bytes of one expert block; 0 if the shape is invalid. */
size_t moe_expert_block_bytes(const moe_expert_shape* shape);
/* Every offset of the block layout described above. */
int moe_expert_block_layout(const moe_expert_shape* shape, moe_block_layout* out);
/* Build one block (host) from the nine canonical arrays (host):
 * q_gate, q_up uint8 [I][H/2]; q_down uint8 [H][I/2] (packed codes);
 * s_gate, z_gate, s_up, z_up fp16 [I][H/g]; s_down, z_down fp16 [H][I/g].
 * Padding bytes are zeroed. */
int moe_pack_expert(const moe_expert_shape* shape,
                    const uint8_t* q_gate, const uint8_t* q_up, const uint8_t* q_down,
                    const uint16_t* s_gate, const uint16_t* z_gate,
                    const uint16_t* s_up, const uint16_t* z_up,
                    const uint16_t* s_down, const uint16_t* z_down,
                    void* block_out);
/* Inverse of moe_pack_expert (host -> host). */
int moe_unpack_expert(const moe_expert_shape* shape, const void* block,
                      uint8_t* q_gate, uint8_t* q_up, uint8_t* q_down,
                      uint16_t* s_gate, uint16_t* z_gate,
                      uint16_t* s_up, uint16_t* z_up,
                      uint16_t* s_down, uint16_t* z_down);

/* ---- routing --------------------------------------------------------------
 * "02 / A solução": the router picks the experts of each token.
 * logits  device fp32 [T][E]  (row-major)
 * ids     device int32 [T][k] out: experts in (logit desc, index asc) order;
 *         -0 == +0, so exact ties go to the lower index.
 * weights device fp32 [T][k] out: p = softmax over all E logits;
 *         w_j = p[id_j] / sum_j' p[id_j'] if renorm, else p[id_j].
 * bad_tokens device int32 [1] or NULL: if non-NULL, incremented (atomically)
 *         once per token whose logits hold NaN or +inf or are all -inf; such a
 *         token gets ids -1 and weights 0 (moe_expert_forward skips id -1).
 * Limits: 1 <= k <= E <= 4096, k <= 32, T >= 0 (T = 0 enqueues nothing).
 */
int moe_route(const float* logits, int T, int E, int k, int renorm,
              int32_t* ids, float* weights, int32_t* bad_tokens, void* stream);

/* ---- token sort -----------------------------------------------------------
 * Groups the (token, choice) pairs p = t*k + j by expert for the grouped
 * executor ("04 / Resultados": compact experts computed in groups).
 * ids      device int32 [T][k]; ids outside [0, E) are dropped.
 * offsets  device int32 [E+1] out: pairs of expert e are [offsets[e], offsets[e+1])
 * pair_tok device int32 [T*k] out: token of each sorted pair
 * pair_j   device int32 [T*k] out: choice index j of each sorted pair
 * Order within an expert: ascending p (stable). Limits: E <= 1024, T*k <= 65536.
 */
int moe_token_sort(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                   int32_t* pair_tok, int32_t* pair_j, void* stream);

/* ---- routed expert FFN ----------------------------------------------------
 * y[t] = sum_j w[t][j] * W_d (silu(W_g x_t) * (W_u x_t))  (+ y_shared[t])
 * with the weights of expert ids[t][j] read from its INT4 block and converted
 * inside the kernel ("03 / Arquitetura", "08 / Comportamento do modelo").
 * x         device fp16 [T][H]
 * ids       device int32 [T][k]; id -1 means "no expert" (contributes 0)
 * weights   device fp32 [T][k]
 * pool      device, n_slots expert blocks back to back ([n_slots][block])
 * slot_of   device int32 [E]: slot of each expert, -1 if not resident
 * y_shared  device fp16 [T][H] or NULL: added to the routed sum (the separate
 *           FP16 non-routed path, "03 / Arquitetura")
 * y         device fp16 [T][H] out (round to nearest even)
 * workspace device, >= moe_forward_workspace_bytes(...) bytes, 256-aligned,
 *           zero-filled before its first use (calls leave it reusable: the
 *           synchronisation counters inside are reset by the call itself;
 *           after a call that set bit 2, zero it again). Calls sharing a
 *           workspace must be ordered (same stream). The GEMV path's blocks
 *           wait on each other (bounded) and so must all be resident at
 *           once: one block per SM, as the library launches them.
 *           Its first 4 bytes are a sticky error word: bit 0 = an id mapped
 *           to a slot outside [0, n_slots) (that pair contributed 0); bit 1 =
 *           an id outside [-1, E); bit 2 = a bounded device wait expired (the
 *           result is not valid). Read it with moe_workspace_flags.
 * path      MOE_PATH_AUTO: GEMV up to 16 tokens and 256 (token, choice) pairs,
 *             else grouped.
 *           MOE_PATH_GEMV: decode dequant-GEMV. One streaming kernel, one
 *             block per SM: the (token, choice) pairs are grouped by expert
 *             so every distinct expert is read once per call; each block
 *             streams its rows of every chosen expert's gate/up and down
 *             sections through shared memory with bulk async copies (both
 *             requested up front), writes h = silu(gate) * up for its rows,
 *             exchanges h with the other blocks through the workspace, and
 *             forms its output rows of the down projection and the top-k
 *             combine. Falls back to the unfused kernels beyond its limits
 *             (H > 4096, I > 2048, more than 16 tokens or 256 pairs,
 *             E > 1024, or shared memory).
 *           MOE_PATH_GROUPED: token-sorted tensor-core grouped GEMM: pairs
 *             sorted by expert, tiles of up to 128 pairs; tcgen05 MMAs with
 *             the expert rows as the 128-row operand (expanded from INT4 to
 *             FP16 in shared memory) and the gathered activations as the
 *             pair operand, FP32 accumulation in tensor memory; then the
 *             down GEMM and a fixed-order combine. Limits: E <= 1024,
 *             T*k <= 65536; y and y_shared 16-byte aligned.
 *           MOE_PATH_GEMV_UNFUSED: the two-kernel dequant-GEMV without the
 *             shared-memory streaming, kept for comparison.
 * Arithmetic: GEMV paths form products in FP16 pairs of at most 8 terms with
 * FP32 accumulation; the grouped path expands each weight to FP16
 * (q - z) * s (one rounding for an integer zero point) and accumulates in
 * FP32 in the tensor cores. All paths round the SwiGLU intermediate to FP16
 * before the down projection.
 */
enum { MOE_PATH_AUTO = 0, MOE_PATH_GEMV = 1, MOE_PATH_GROUPED = 2, MOE_PATH_GEMV_UNFUSED = 3 };
size_t moe_forward_workspace_bytes(const moe_expert_shape* shape, int T, int k,
                                   int E, int path);
int moe_expert_forward(const moe_expert_shape* shape, const void* x, int T,
                       const int32_t* ids, const float* weights, int k, int E,
                       const void* pool, const int32_t* slot_of, int n_slots,
                       const void* y_shared, void* y, void* workspace,
                       size_t workspace_bytes, int path, void* stream);
/* ---- routed expert FFN reading absent experts over the CPU-GPU link -------
 * moe_expert_forward's result, computed by the two-kernel dequant-GEMV
 * (MOE_PATH_GEMV_UNFUSED), where an expert whose slot_of entry is -1 is
 * not skipped but read in place, by the kernels' own loads, from the layer's
 * complete host source: a weight that is not in the right memory is read
 * again at every use (lucashiago.com.br "local" explainer, etapa 5, whose
 * time model t_token = t_calc + bytes_out / bandwidth prices it). No copy
 * engine, slot change or host round trip is involved, so a whole decode step
 * can be enqueued (or captured in a graph) without waiting for routing.
 * host_src  host [E][block] of this layer, page-locked and mapped into the
 *           device address space (cudaHostAlloc, or cudaHostRegister on a
 *           unified-addressing system), 16-byte aligned; read only. Not
 *           page-locked or not mapped: MOE_ERR_ARG.
 * Entries of slot_of at or above n_slots still set bit 0 of the error word
 * and contribute 0. Other arguments and limits as moe_expert_forward.
 */
int moe_expert_forward_zero_copy(const moe_expert_shape* shape, const void* x, int T,
                                 const int32_t* ids, const float* weights, int k, int E,
                                 const void* pool, const int32_t* slot_of, int n_slots,
                                 const void* host_src, const void* y_shared, void* y,
                                 void* workspace, size_t workspace_bytes, void* stream);
/* ---- routed layer: routing + expert FFN in one call ----------------------
 * The same result as moe_route(logits, ...) followed by
 * moe_expert_forward(...): the router picks each token's experts and their
 * weights ("02 / A solução") and the chosen INT4 experts run on x. On the
 * GEMV path (MOE_PATH_GEMV, or MOE_PATH_AUTO at T <= 16 and T*k <= 256) with
 * the streamed decode kernel's limits (H <= 4096, inter <= 2048, E <= 1024)
 * the routing runs inside that kernel: every block picks the same experts
 * with moe_route's selection and fixed-order softmax (one token: the block's
 * producer warp; several: a warp per token), so no separate routing kernel
 * or id round trip sits between the layer's input and its weight stream;
 * otherwise moe_route runs first.
 * logits  device fp32 [T][E]; ids / weights device out [T][k] (the routing
 * used, as moe_route defines it: NaN/+inf/all -inf tokens get ids -1).
 * Other arguments as moe_expert_forward; limits as moe_route.
 */
int moe_layer_forward(const moe_expert_shape* shape, const void* x, const float* logits, int T,
                      int E, int k, int renorm, int32_t* ids, float* weights, const void* pool,
                      const int32_t* slot_of, int n_slots, const void* y_shared, void* y,
                      void* workspace, size_t workspace_bytes, int path, void* stream);
/* ---- routed layer without any device allocation --------------------------
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory: plugins and serving runtimes whose host
 * framework owns every device allocation and forbids extra ones, and
 * deployments with a fixed, pre-planned memory budget.
 * Same arguments and result as moe_layer_forward on the MOE_PATH_GEMV path,
 * minus the workspace: the scratch it needs (a header with the error word and
 * the kernel's counters, then the FP16 SwiGLU intermediate of every
 * (token, choice) pair) lives in a 1 MiB array compiled into the library,
 * held by every GPU that loads the library until the process exits. The call
 * allocates nothing (no cudaMalloc/cudaFree); it clears the header with one
 * cudaMemsetAsync on `stream` before the kernel.
 * Limits: 256 + ceil(4*T*k / 256)*256 + T*k*inter*2 bytes <= 1 MiB, else
 * MOE_ERR_CAPACITY (at inter 1024 about 500 pairs; the kernel's own limits
 * below come first); H <= 4096, inter <= 2048, T <= 16, T*k <= 256 and
 * E <= 1024 (the streamed decode kernel), else MOE_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it. The cached address belongs to the
 * device's current context: after cudaDeviceReset the library must be
 * reloaded (or the process restarted) before this call is used again on that
 * device. Nothing is stated here about capturing this call in a CUDA graph.
 * Every call shares the one array: calls that overlap on the GPU (different
 * streams, or other threads) race and corrupt each other's results; order
 * them on one stream. Each call keeps its error word (bit 0: an id without a
 * slot, bit 1: an id outside [-1, E), bit 2: a bounded device wait expired and
 * y is not valid) until the next call clears it: read it with
 * moe_layer_forward_noalloc_flags.
 */
int moe_layer_forward_noalloc(const moe_expert_shape* shape, const void* x, const float* logits,
                              int T, int E, int k, int renorm, int32_t* ids, float* weights,
                              const void* pool, const int32_t* slot_of, int n_slots,
                              const void* y_shared, void* y, void* stream);
/* The error word of the last moe_layer_forward_noalloc call on the current
 * device (bits as above) into *flags_out (host): one cudaMemcpyAsync on
 * `stream`, then a synchronisation of `stream`. No allocation. */
int moe_layer_forward_noalloc_flags(int32_t* flags_out, void* stream);
/* Clear (zero) the workspace error word: enqueued on `stream`. */
int moe_workspace_clear_flags(void* workspace, void* stream);
/* Read the workspace error word into *flags_out: synchronises `stream`. */
int moe_workspace_flags(const void* workspace, int32_t* flags_out, void* stream);

/* ---- shared (non-routed) FP16 SwiGLU FFN ----------------------------------
 * y = W_d (silu(W_g x) * (W_u x)) with FP16 weights ("03 / Arquitetura": the
 * non-routed parts stay FP16).
 * x  device fp16 [T][H]; wg, wu device fp16 [Is][H]; wd device fp16 [H][Is];
 * y  device fp16 [T][H] out. workspace >= moe_shared_workspace_bytes(T, H, Is),
 *    256-aligned, zero-filled before its first use; its first 4 bytes are the
 *    sticky error word (bit 2: a bounded device wait expired), then h [T][Is].
 * Two tcgen05 GEMM kernels (gate/up with the SwiGLU epilogue, then down):
 * operands by TMA, FP32 accumulation in tensor memory, h and y rounded to
 * FP16. Limits: H, Is positive multiples of 64 (<= 65536); x, weights and y
 * 16-byte aligned. Errors: MOE_ERR_ARG (shape, NULL, alignment),
 * MOE_ERR_CAPACITY (workspace too small), MOE_ERR_CUDA.
 */
size_t moe_shared_workspace_bytes(int T, int H, int Is);
int moe_shared_forward(const void* x, int T, int H, int Is, const void* wg,
                       const void* wu, const void* wd, void* y, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---- residency manager ----------------------------------------------------
 * Per-layer GPU slot pools fed from a complete, immutable host source
 * ("03 / Arquitetura", ADR 0009). One decode step of one layer:
 *   1. every count c of the layer becomes c*decay, then gains 1 per id given;
 *   2. N = distinct ids; |N| > slots is MOE_ERR_CAPACITY (nothing changes);
 *   3. misses N \ resident, in ascending id order; when the resident set is
 *      full a victim leaves it (policy below); the miss takes the lowest free
 *      slot (a spare) else the victim's slot;
 *   4. each miss is copied host->device with cudaMemcpyAsync on the copy
 *      stream, after the copy stream waited for every reader of the slot
 *      enqueued so far on the compute stream;
 *   5. the compute stream waits for the copies, then a one-block kernel
 *      publishes the new slot table [E] of the layer (the new generation).
 * Initial state: expert e in slot e for e < slots ("canonical initial
 * placement"), counts 0, spare slots free.
 * Victim policies (the candidates are resident \ N):
 *   MOE_POLICY_DECAY   argmin (decayed count, id): an access counter whose
 *                      old accesses lose weight (Strata page);
 *   MOE_POLICY_LRU     argmin (step of last use, id), never-used = -1: the
 *                      evolving LRU of the claims.json experiment contract;
 *   MOE_POLICY_PINNED  the `pinned` experts of each layer with the highest
 *                      `profile` value (ties: lower id) are resident from the
 *                      start and never evicted; the other slots follow LRU
 *                      (lucashiago.com.br "local" explainer, etapa 4: a
 *                      profile fixes yesterday's popular set, LRU adapts).
 *                      Initial resident set: the pinned experts plus the
 *                      lowest other ids, in slots 0.. by ascending id.
 *                      Requires pinned <= slots - min(max_ids_per_step, E).
 */
enum { MOE_POLICY_DECAY = 0, MOE_POLICY_LRU = 1, MOE_POLICY_PINNED = 2 };
typedef struct {
  int32_t layers;            /* L */
  int32_t experts;           /* E per layer */
  int32_t slots;             /* C: experts resident per layer (1..E) */
  int32_t spares;            /* S: extra physical slots per layer (>= 0) */
  int32_t max_ids_per_step;  /* upper bound on n passed to prepare */
  int32_t dry_run;           /* 1: decide and trace only, no CUDA work */
  uint64_t block_bytes;      /* bytes of one expert block */
  double decay;              /* count decay per step, in (0, 1] */
  int32_t policy;            /* MOE_POLICY_* (0: decayed counts) */
  int32_t pinned;            /* MOE_POLICY_PINNED: experts pinned per layer */
  const double* profile;     /* MOE_POLICY_PINNED: host [L][E] popularity, read by create */
  int32_t log_ops;           /* 1: keep a log of the stream operations (moe_residency_ops) */
} moe_residency_cfg;

typedef struct {
  uint64_t steps, hits, misses, evictions, copies, h2d_bytes;
  uint64_t prefetched;       /* misses served by a prefetched copy (no copy in their step) */
  uint64_t prefetch_copies;  /* copies made by moe_residency_prefetch */
} moe_residency_stats;

typedef struct {
  int64_t step;    /* prepare() calls made on this layer before this one */
  int32_t layer;
  int32_t expert;  /* the miss */
  int32_t slot;    /* physical slot it was copied into */
  int32_t victim;  /* evicted expert, -1 if none */
} moe_residency_event;

/* One stream operation of the manager, in the order it was enqueued. Streams:
 * 0 compute, 1 copy. Events: 0 "readers done" (compute), 1 "copies done"
 * (copy). The log is the same in a dry run, which
 * enqueues nothing, so the ordering can be checked without a GPU. */
enum { MOE_OP_RECORD = 0, MOE_OP_WAIT = 1, MOE_OP_COPY = 2, MOE_OP_PUBLISH = 3 };
typedef struct {
  int32_t kind;    /* MOE_OP_*: RECORD event on stream, stream WAITs for event, COPY, PUBLISH */
  int32_t stream;  /* 0 compute, 1 copy */
  int32_t event;   /* RECORD / WAIT; else -1 */
  int32_t layer;   /* COPY / PUBLISH; else -1 */
  int32_t slot;    /* COPY: destination slot; else -1 */
  int32_t expert;  /* COPY: the expert copied; else -1 */
} moe_residency_op;

typedef struct moe_residency moe_residency;

/* host_src: host [L][E][block_bytes], page-locked (cudaHostAlloc /
 *   cudaHostRegister), owned by the caller, never written by the library,
 *   must outlive the handle.
 * dev_pool: device [L][slots+spares][block_bytes]; dev_slot_of: device
 *   int32 [L][E]. Both owned by the caller. create() fills the pool with the
 *   canonical placement and the slot table, synchronously.
 * compute, copy: cudaStream_t. Capacity errors (slots > E, max_ids_per_step
 *   distinct experts not fitting) return MOE_ERR_CAPACITY and no handle. */
int moe_residency_create(const moe_residency_cfg* cfg, const void* host_src,
                         void* dev_pool, int32_t* dev_slot_of, void* compute,
                         void* copy, moe_residency** out);
/* host_ids: host int32 [n], the ids all tokens of this step need in `layer`
 * (entries outside [0, E) are rejected with MOE_ERR_ARG, state unchanged). */
int moe_residency_prepare(moe_residency* r, int layer, const int32_t* host_ids, int n);
/* Prefetch of predicted misses into spare slots ("03 / Arquitetura", ADR
 * 0009: a copy lands in a spare position while readers keep the current
 * generation). For each id in order, skipping ids that are resident or
 * already prefetched, while a free spare slot is left: the block is copied
 * host->device on the copy stream into the lowest free slot. Nothing is
 * published and no count changes. The copy adds no wait: a free slot was
 * never read, or was freed by a prepare() whose copy-stream wait already
 * follows every reader of its previous occupant (the copy stream runs in
 * order), so it overlaps the layers being computed. The layer's next prepare() takes a prefetched
 * expert that its step needs as a miss in that slot, with no copy (counted
 * in `prefetched`); prefetched experts that step does not need return to
 * the free spares. Returns the number copied in *staged_out (nullable).
 * Ids outside [0, E): MOE_ERR_ARG, nothing staged. */
int moe_residency_prefetch(moe_residency* r, int layer, const int32_t* host_ids, int n, int* staged_out);
/* layer = -1 sums over layers. */
int moe_residency_get_stats(const moe_residency* r, int layer, moe_residency_stats* out);
/* Copies up to `cap` events (all layers, in decision order); *n_out = total. */
int moe_residency_trace(const moe_residency* r, moe_residency_event* buf,
                        size_t cap, size_t* n_out);
/* Copies up to `cap` logged stream operations (cfg.log_ops); *n_out = total. */
int moe_residency_ops(const moe_residency* r, moe_residency_op* buf, size_t cap, size_t* n_out);
/* Host copy of the layer's current slot table [E] (what was last published). */
int moe_residency_slot_table(const moe_residency* r, int layer, int32_t* host_out);
/* Host copy of the layer's decayed counts [E]. */
int moe_residency_counts(const moe_residency* r, int layer, double* host_out);
/* Test hook: the nth copy enqueue from now (0-based) fails with
 * MOE_ERR_INJECTED before it is issued; -1 disables. On such a failure the
 * step is not published: counts, slot table and statistics keep their
 * previous values, except that an expert whose slot was already overwritten
 * by an earlier copy of the failed step (no spare was free) is marked absent
 * and that removal is published. */
int moe_residency_inject_copy_failure(moe_residency* r, int64_t nth_copy);
/* Waits for the handle's copies, frees its events. NULL is a no-op. */
void moe_residency_destroy(moe_residency* r);

#ifdef __cplusplus
}
#endif

#endif /* INT4_ROUTED_EXPERT_MOE_GB300_MOE_H */
