/*
 * mq.h -- C ABI of libmq, the GB300 (sm_103a) q4_K x q8_0 decode matvec.
 *
 * What the library computes (pages: "07 . R3 -- Small-model per-token
 * overhead" section 1 for MMVQ = dp4a x q8_0 on q4_K weights; "04 . 8o --
 * Killing the CPU stall at decode start" sections 1, 3.1 and 3.2 for the
 * concatenated gate/up weight ffn_gu and the row-concat preconditions;
 * "Part 4 . Lecture 08 -- Graph-Resident Decode" sections 2-4 for shapes and
 * pointers held in device memory, grid sizes as capture keys and lazy state
 * pre-warmed before capture):
 *
 *   xq = q8_0(x)                          32-value blocks, f16 scale
 *   y  = W . xq                           W rows of 256-weight q4_K super-blocks
 *   h  = SiLU(W_gu[0:I] . xq) * (W_gu[I:2I] . xq);  y = W_down . q8_0(h)
 *   step = for each layer: qkv, o, FFN, in that order, on one stream
 *
 * Formats (the pages name them; the bytes are the GGUF-compatible reading):
 *   q4_K super-block, 256 weights, 144 bytes: [0:2] d f16, [2:4] dmin f16,
 *     [4:16] eight 6-bit scale/min pairs, [16:144] 4-bit quants; weight =
 *     d*sc*q - dmin*m.  A row of K weights is K/256 blocks, K % 256 == 0.
 *   q8_0 block, 32 values, 34 bytes: [0:2] f16 scale d = amax/127 (fp32 IEEE
 *     division, then round-to-nearest-even to f16), [2:34] int8
 *     round_half_away(x/d).
 *
 * Layouts: matrices are row-major with dense rows (row stride = K/256*144
 * bytes).  Multi-column activations are column-major by token: column c of an
 * fp32 input is x[c*K .. c*K+K), of a q8_0 input the bytes
 * [c*K/32*34, (c+1)*K/32*34); column c of an output is y[c*y_ld .. +rows).
 *
 * Ownership: the caller allocates and owns every buffer (weights, inputs,
 * outputs, descriptors, the FFN's h_q8 scratch).  After mq_init the library
 * allocates nothing, never synchronizes inside a compute call and never reads
 * device memory from the host, so every compute call can be captured into a
 * CUDA graph.  Weights must stay unchanged while a graph that reads them lives.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  Every compute call is asynchronous on that stream.
 *
 * Errors: each call returns an mq_status.  Host-side checks run before any
 * launch; a call that fails them launches nothing.  A failed CUDA launch
 * returns MQ_ERR_CUDA and mq_last_cuda_error() gives the cudaError_t.  Kernels
 * re-check the device descriptor against the host-side shapes they were
 * sized for; on a mismatch they write nothing and record the problem in the
 * device status word (mq_read_device_status).  Nothing aborts, throws or exits.
 */
#ifndef MQ_H
#define MQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MQ_ABI_VERSION 3

typedef int mq_status;
#define MQ_OK 0
#define MQ_ERR_INVALID_ARG 1     /* null pointer, unknown type, bad count */
#define MQ_ERR_SHAPE 2           /* K % 256 (q4_K) or K % 32 (q8_0), ncols outside 0..8, negative sizes */
#define MQ_ERR_ALIGN 3           /* a pointer is not aligned as its layout requires */
#define MQ_ERR_CUDA 4            /* a CUDA call failed; see mq_last_cuda_error */
#define MQ_ERR_UNSUPPORTED 5     /* size beyond the library's limits (see MQ_MAX_*) */
#define MQ_ERR_NOT_INITIALIZED 6 /* mq_init was not called for the current device */

/* device status word bits (mq_read_device_status) */
#define MQ_DEV_DESC_MISMATCH 1u  /* a kernel's device descriptor disagreed with its launch shape */
#define MQ_DEV_DESC_ALIGN 2u     /* a device descriptor held a misaligned pointer */
#define MQ_DEV_TIMEOUT 4u        /* a kernel's bounded wait on its copy pipeline gave up; outputs not written */
#define MQ_DEV_ALIAS 8u          /* a persistent step's input overlaps an output of the same launch outside
                                    the MQ_STEP_CHAINED pattern; nothing was written */

/* quantization types (mq_concat_rows*) */
#define MQ_TYPE_Q4_K 1
#define MQ_TYPE_Q8_0 2
#define MQ_TYPE_Q4_0 3  /* 32 weights in 18 bytes: f16 d, 16 bytes of nibbles (see mq_matvec_q4_0_q8_0) */

/* limits: K * ncols <= MQ_MAX_K_TIMES_NCOLS (the q8_0 activation is staged in
 * shared memory), K <= MQ_MAX_K, ncols <= MQ_MAX_NCOLS */
#define MQ_MAX_NCOLS 8
#define MQ_MAX_K 131072
#define MQ_MAX_K_TIMES_NCOLS 163840

const char* mq_status_string(mq_status s);
int mq_abi_version(void);
/* cudaError_t of the last CUDA failure seen by this thread (0 if none) */
int mq_last_cuda_error(void);

/* Pre-warm everything a compute call would otherwise do lazily: device
 * properties, shared-memory opt-ins of every kernel, the device status word.
 * Call once per device, outside any stream capture, before other calls.
 * Leaves the caller's current device unchanged. */
mq_status mq_init(int device);

/* Read the device status word of the current device and reset it to zero.
 * Synchronizes `stream`; not for use inside a capture. */
mq_status mq_read_device_status(uint32_t* bits, void* stream);

/* ---- sizes (pure host) ---------------------------------------------------- */
/* bytes of one q4_K row of K weights: K/256*144 (0 if K % 256 != 0) */
size_t mq_q4K_row_bytes(int64_t K);
/* bytes of one q8_0 column of K values: K/32*34 (0 if K % 32 != 0) */
size_t mq_q8_0_bytes(int64_t K);
/* elements and bytes per block of a type (0 for an unknown type) */
int mq_quant_block_elems(int32_t ttype);
int mq_quant_block_bytes(int32_t ttype);

/* ---- row concatenation ("04 . 8o", section 3.2) ----------------------------
 * Feasible iff n >= 2, every tensor has type ttype[0], the same ne0, ne0 is a
 * multiple of the type's block size, and each tensor's byte length equals
 * ne1 * (ne0/block_elems) * block_bytes.  Reads the metadata only.
 * Returns 1 if feasible, 0 otherwise (also for null arrays). */
int mq_concat_rows_feasible(int32_t n, const int32_t* ttype, const int64_t* ne0,
                            const int64_t* ne1, const uint64_t* nbytes);
/* dst = rows of srcs[0], then srcs[1], ...; device pointers; the same
 * preconditions as mq_concat_rows_feasible (checked with nbytes computed from
 * rows).  Device-to-device copies on `stream`.  Builds ffn_gu (gate rows then
 * up rows) and the q|k|v projection. */
mq_status mq_concat_rows(void* dst, const void* const* srcs, const int64_t* rows, int32_t n,
                         int32_t ttype, int64_t ne0, void* stream);

/* ---- q8_0 quantization -----------------------------------------------------
 * x: fp32 [ncols][K] device, 4-byte aligned; xq: q8_0 [ncols][K/32] blocks,
 * 2-byte aligned.  K % 32 == 0.  ncols == 0 or K == 0 launches nothing. */
mq_status mq_quantize_q8_0(const float* x, void* xq, int64_t K, int32_t ncols, void* stream);

/* ---- matvec ------------------------------------------------------------------
 * Device-resident descriptor (caller-allocated, 8-byte aligned).  The kernel
 * reads it at start, so a captured graph follows any change made to it
 * between replays, as long as the shapes stay those the launch was sized for.
 *   W      q4_K [rows][K/256] super-blocks, 16-byte aligned
 *   x      fp32 [ncols][K], 4-byte aligned, or NULL; when set the kernel
 *          quantizes it to q8_0 itself (bit-identical to mq_quantize_q8_0)
 *   xq     q8_0 [ncols][K/32], 2-byte aligned; read when x == NULL
 *   xq_out nullable; when x is set, the q8_0 of x is also written here
 *   y      fp32 [ncols][y_ld], 4-byte aligned, y_ld >= rows
 */
typedef struct mq_mv_desc {
    const void* W;
    const float* x;
    const void* xq;
    void* xq_out;
    float* y;
    int32_t rows;
    int32_t K;
    int32_t ncols;
    int32_t y_ld;
} mq_mv_desc;

/* host-side validation of a host copy of a descriptor (shapes, alignment, nulls) */
mq_status mq_check_mv_desc(const mq_mv_desc* h_desc);
/* y[c][r] = sum over K of W[r] . q8_0(x)[c], fp32 output.  rows, K, ncols are
 * the host copies of the descriptor's shapes: they size the grid (the capture
 * key) and must equal the device descriptor's.  rows == 0 or ncols == 0
 * launches nothing; K must be a positive multiple of 256.  Where the whole
 * staged activation does not fit beside the weight ring (e.g. 8 columns of
 * K = 18944), the call runs as 2..4 launches in stream order, each over an
 * equal part of every row, the later ones adding to y (y = part 0 + part 1
 * + ..., in that order); a captured graph then holds one kernel per part. */
mq_status mq_matvec_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols,
                             void* stream);

/* ---- the matvec for the other weight types -------------------------------------
 * The pages' 0.5B model is quantized q4_0 ("07 . R3 -- Small-model per-token
 * overhead", sections 4 and 5); the same MMVQ dot product against q8_0
 * activations serves q4_0 and q8_0 weights (GGUF-compatible layouts):
 *   q4_0: 32 weights in 18 bytes: [0:2] f16 d, [2:18] byte i holds weight i
 *         in its low nibble and weight i+16 in its high nibble; w = d*(q-8).
 *   q8_0: 32 weights in 34 bytes, the activation's block format; w = d*q.
 * Same descriptor, shapes, limits and rules as mq_matvec_q4K_q8_0, with W of
 * rows x K/32 blocks of that type (row bytes K/32*18 or K/32*34); K % 256 ==
 * 0 so rows stay 16-byte multiples.  These run only on the bulk-copy ring
 * kernels: a shape whose ring plan does not fit the device returns
 * MQ_ERR_UNSUPPORTED. */
mq_status mq_matvec_q4_0_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* stream);
mq_status mq_matvec_q8_0_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* stream);

/* ---- fused FFN -----------------------------------------------------------------
 *   W_gu   q4_K [2I][H]: gate rows 0..I-1, then up rows I..2I-1 (ffn_gu)
 *   W_down q4_K [H][I]
 *   x      fp32 [ncols][H] or NULL (then xq q8_0 [ncols][H/32] is read)
 *   h_q8   q8_0 [ncols][I/32]: scratch written by the gate/up kernel and read
 *          by the down kernel (caller-owned, 2-byte aligned)
 *   gu_dbg nullable fp32 [ncols][2I]: g then u, as the kernel computed them
 *   h_dbg  nullable fp32 [ncols][I]: SiLU(g)*u before its re-quantization
 *   y      fp32 [ncols][y_ld], y_ld >= H
 * H % 256 == 0 and I % 256 == 0. */
typedef struct mq_ffn_desc {
    const void* W_gu;
    const void* W_down;
    const float* x;
    const void* xq;
    void* h_q8;
    float* gu_dbg;
    float* h_dbg;
    float* y;
    int32_t H;
    int32_t I;
    int32_t ncols;
    int32_t y_ld;
} mq_ffn_desc;

mq_status mq_check_ffn_desc(const mq_ffn_desc* h_desc);
/* Two launches on `stream`: (1) g|u = W_gu . q8_0(x), h = SiLU(g)*u, h_q8 =
 * q8_0(h) in the epilogue; (2) y = W_down . h_q8 (split over K like the
 * matvec where h does not fit beside the ring).  The down launch uses
 * programmatic dependent launch: its weight copies start while (1) drains, and
 * it reads h only after its grid-dependency wait. */
mq_status mq_ffn_gu_silu_down(const mq_ffn_desc* d_desc, int32_t H, int32_t I, int32_t ncols,
                              void* stream);
/* The first of those two launches alone: fills h_q8 (and the debug outputs),
 * leaves y untouched.  W_down and y may be NULL in the descriptor. */
mq_status mq_ffn_gate_up(const mq_ffn_desc* d_desc, int32_t H, int32_t I, int32_t ncols, void* stream);

/* ---- whole decode step of a layer stack ------------------------------------------
 * Per layer, in order: qkv (the concatenated q|k|v projection, input x = a_l),
 * o (input b_l), then the FFN (input c_l).  d_layers: device array of
 * n_layers layer descriptors.  h_shape: host copy of the shapes (grid sizes;
 * the capture key).  Capturable as one CUDA graph.
 *
 * A stack of FFN layers only: qkv_rows == 0 and o_rows == 0 (then o_K and the
 * qkv and o parts of every descriptor are ignored); either projection may be
 * left out on its own the same way. */
typedef struct mq_layer_desc {
    mq_mv_desc qkv;
    mq_mv_desc o;
    mq_ffn_desc ffn;
} mq_layer_desc;

#define MQ_STEP_PDL 1u         /* multi-kernel path: launch with programmatic dependent launch */
#define MQ_STEP_PERSISTENT 2u  /* one persistent kernel for the whole stack (needs `workspace`) */
#define MQ_STEP_CHAINED 4u     /* every phase reads the previous phase's output (a real decode chain) */

/* bytes of the persistent step's fixed workspace words (abort word, phase
 * counter, a reserved word per CTA); the whole workspace a shape needs is
 * mq_step_workspace_bytes */
#define MQ_STEP_WORKSPACE_BYTES 4352

typedef struct mq_step_shape {
    int32_t n_layers;
    int32_t H;        /* hidden: K of qkv and of ffn_gu, rows of down */
    int32_t I;        /* intermediate */
    int32_t qkv_rows; /* rows of the q|k|v matrix */
    int32_t o_rows;   /* rows of o */
    int32_t o_K;      /* K of o */
    int32_t ncols;
    uint32_t flags;   /* MQ_STEP_* */
    void* workspace;  /* MQ_STEP_PERSISTENT: caller-owned device memory of
                         mq_step_workspace_bytes(shape) bytes, 16-byte
                         aligned; zeroed by the call on its stream (so a
                         captured graph re-zeroes it every replay); two steps
                         that overlap on the GPU must not share it */
} mq_step_shape;

/* Without MQ_STEP_PERSISTENT: four launches per layer (qkv, o, gate/up, down).
 * With it: a single cooperative launch of one CTA per SM that runs every
 * layer, the weight stream running ahead across the dependency points.  At
 * each point a CTA waits, bounded in time (a timeout records MQ_DEV_TIMEOUT),
 * until what it reads has been written.  The gate/up phase writes h into
 * `workspace` as tagged records (a data word and its phase in one 8-byte
 * store), which the down phase reads and checks word by word.  Both paths give
 * bit-identical outputs.  The persistent kernel needs every SM: it fails with
 * MQ_ERR_CUDA if the device cannot host its whole grid at once.  It returns
 * MQ_ERR_UNSUPPORTED where its shared memory cannot hold a phase's whole
 * activation beside its weight ring (H = 3584, I = 18944 from 4 columns on); the
 * four-launch form runs those shapes.
 *
 * Inputs of the persistent step:
 *  - default: every input (a_l, b_l, c_l or their q8_0 forms) is a buffer that
 *    no phase of the launch writes.  Each CTA adds one to a phase counter once
 *    it has written a phase's outputs and the next phase waits until the
 *    counter shows every CTA, which orders the phases; no input is produced in
 *    the launch, so no input needs to be made visible.  The kernel checks every input against
 *    every output of the launch first; an overlap records MQ_DEV_ALIAS and
 *    nothing is written.
 *  - MQ_STEP_CHAINED: a decode chain.  The input of every qkv, o and FFN phase
 *    is the fp32 output of the phase before it: o_l.x == qkv_l.y, ffn_l.x ==
 *    o_l.y, qkv_{l+1}.x == ffn_l.y (with a phase left out, the one before
 *    it); layer 0's first phase reads the caller's input.  For ncols > 1 the
 *    producer's y_ld must equal the consumer's K.  Every such output is also
 *    written into `workspace` as tagged records, and the consumer stages its
 *    input from them, so one load both reads a value and proves it written
 *    (no fence on the path).  The kernel checks the pattern first; a
 *    descriptor that breaks it records MQ_DEV_DESC_MISMATCH and nothing is
 *    written.  Without MQ_STEP_PERSISTENT the flag changes nothing: kernel
 *    boundaries order the launches whatever the inputs are. */
mq_status mq_step(const mq_layer_desc* d_layers, const mq_step_shape* h_shape, void* stream);

/* Bytes of workspace mq_step needs for h_shape with MQ_STEP_PERSISTENT (and
 * the shape's flags): MQ_STEP_WORKSPACE_BYTES plus ncols * (I/128) * 320
 * bytes of h records, and with MQ_STEP_CHAINED 8 * ncols * rows bytes of
 * output records for each of q|k|v, o and down that is present (rows =
 * qkv_rows, o_rows, H), each rounded up to a multiple of 32.  Host only; checks the shape as mq_step does
 * (MQ_ERR_SHAPE, and MQ_ERR_INVALID_ARG for a null pointer).  The call cannot
 * see the workspace's size: a smaller workspace is the caller's error. */
mq_status mq_step_workspace_bytes(const mq_step_shape* h_shape, size_t* bytes);

/* ---- more columns: the q4_K x q8_0 matmul on the tensor cores ("MMQ") ----------------
 * "07 . R3 -- Small-model per-token overhead", section 5: past the decode
 * matvec the engine's next work was MMQ, the quantized matmul for more
 * tokens.  y[c][r] = sum over K of W[r] . q8_0(x)[c] for 1..MQ_MMQ_MAX_NCOLS
 * columns (meant for 9 and more; the decode kernels serve 1..8), the same
 * descriptor and result as mq_matvec_q4K_q8_0: the q8_0 codes and every
 * 32-element sub-block's integer sum are exact (binary16 operands of the
 * tensor-core MMA, fp32 accumulation of integers below 2^24), and the scales
 * are applied per sub-block in fp32.  Float results match the oracle within
 * the same tolerance as the decode kernels (not bit for bit: the order of the
 * float operations differs).
 *   workspace: caller-owned device memory, 128-byte aligned, of at least
 *   mq_mmq_workspace_bytes(rows, K, ncols) bytes (the activation laid out for
 *   the MMA, and partial sums when a matrix has few 128-row tiles); two calls
 *   that overlap on the GPU must not share it.
 * Three launches at most on `stream` (activation, matmul, partial sums).
 * MQ_ERR_INVALID_ARG for a workspace smaller than needed. */
#define MQ_MMQ_MAX_NCOLS 64
mq_status mq_mmq_workspace_bytes(int32_t rows, int32_t K, int32_t ncols, size_t* bytes);
mq_status mq_mmq_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols, void* workspace,
                          size_t ws_bytes, void* stream);

/* ---- prefill: the resident f16 weight cache and the tensor-core GEMM -----------------
 * "07 . R3 -- Small-model per-token overhead", section 1: 7B prefill at 2K
 * tokens runs a half-precision tensor-core GEMM over a resident f16 copy of
 * the quantized weights, built once.
 *
 * mq_dequant_q4K_f16: W16[r][k] = f16(d*sc*q - dmin*m) of q4_K W [rows][K/256]
 *   (the weight formed exactly, rounded once to nearest-even); W 16-byte
 *   aligned, W16 f16 [rows][K] 16-byte aligned, K % 256 == 0.
 * mq_convert_f32_f16: y[i] = f16(x[i]) (round to nearest-even), n values;
 *   x 4-byte, y 2-byte aligned.
 * mq_gemm_f16: Y[t][r] = sum over k of X16[t][k] * W16[r][k], fp32
 *   accumulation on the tensor cores (tcgen05), fp32 Y [T][R] (row t of Y
 *   holds token t's R outputs).  W16 [R][K] and X16 [T][K] f16 row-major,
 *   16-byte aligned; Y 4-byte aligned; K % 64 == 0; R, T >= 1.  Unlike the
 *   decode calls the operands' addresses are baked into the launch (tensor
 *   maps built on the host), so a captured graph keeps the buffers it saw.
 *   Limits: K <= MQ_MAX_K. */
mq_status mq_dequant_q4K_f16(const void* W, void* W16, int64_t rows, int64_t K, void* stream);
mq_status mq_convert_f32_f16(const float* x, void* y, int64_t n, void* stream);
mq_status mq_gemm_f16(const void* W16, const void* X16, float* Y, int32_t R, int32_t K, int32_t T, void* stream);

/* ---- the FFN without caller scratch --------------------------------------------------
 * No counterpart in the pages: they describe the FFN kernels, not how a
 * caller supplies their scratch.  This entry point exists for callers that
 * cannot allocate device memory for the h_q8 scratch (and the descriptor)
 * that mq_ffn_gu_silu_down takes: a plugin or custom-op hook inside a host
 * runtime that owns every device allocation, or an engine that has handed
 * all free HBM to its cache pool.  It computes the same result as
 * mq_ffn_gu_silu_down with the same kernels (bit-identical y), taking plain
 * device pointers instead of a device descriptor:
 *   W_gu q4_K [2I][H], W_down q4_K [H][I], x fp32 [ncols][H] or NULL (then
 *   xq q8_0 [ncols][H/32] is read), y fp32 [ncols][y_ld], y_ld >= H;
 *   the same shape and alignment rules as mq_check_ffn_desc.
 * Scratch: a fixed device array inside the library, one per device, holding
 * the descriptor and h_q8.  The call allocates nothing (no cudaMalloc, no
 * allocating library routine); it launches three kernels on `stream`: one
 * that writes the descriptor into that array, then the gate/up and the down
 * kernels.  Nothing in the array has to start at zero: every call rewrites
 * the descriptor, and the gate/up kernel writes every h_q8 byte that the down
 * kernel reads.
 * Limit: ncols * (I/32) * 34 bytes of h_q8 must not exceed
 * MQ_NOALLOC_HQ8_MAX_BYTES; larger calls return MQ_ERR_UNSUPPORTED before
 * any device work (use mq_ffn_gu_silu_down with caller scratch for them).
 * Setup: mq_init looks up that device's copy of the array once and caches
 * its address; the call itself only reads the cached address.  Needs mq_init
 * for the device.
 * Races: every call on one device uses the same array, so two calls that
 * overlap on the GPU (two streams, two host threads, or a call in flight
 * while another runs) race on it and give wrong results; order them on one
 * stream or by events. */
#define MQ_NOALLOC_HQ8_MAX_BYTES 131072
mq_status mq_ffn_gu_silu_down_noalloc(const void* W_gu, const void* W_down, const float* x, const void* xq,
                                      float* y, int32_t H, int32_t I, int32_t ncols, int32_t y_ld,
                                      void* stream);

/* ---- test export ---------------------------------------------------------------------
 * The per-32-block integer sums of a matvec, computed by the same device code
 * as the matvec kernel: sumi int32 [ncols][rows][K/32] = sum q4*q8 per block,
 * sumq int32 [ncols][K/32] = sum q8 per block. */
mq_status mq_debug_block_sums_q4K_q8_0(const mq_mv_desc* d_desc, int32_t rows, int32_t K, int32_t ncols,
                                       int32_t* sumi, int32_t* sumq, void* stream);

/* Test-only setter of the kernel family used by later calls (process-wide,
 * not thread-safe): MQ_VARIANT_AUTO (default) uses the bulk-copy ring kernels
 * wherever their shared-memory plan fits and the register-streaming kernels
 * elsewhere; MQ_VARIANT_FORCE_REGISTER always uses the register-streaming
 * kernels.  Both give results within the same tolerance; a graph captured
 * under one setting keeps it. */
#define MQ_VARIANT_AUTO 0
#define MQ_VARIANT_FORCE_REGISTER 1
mq_status mq_debug_set_variant(int32_t policy);

/* Test-only fault injection for later calls (process-wide, not thread-safe).
 * MQ_FAULT_WITHHOLD_TILE: in the bulk-copy ring kernels the producer never
 * delivers each CTA's last tile and every wait is limited to 50 ms, so the
 * consumers' bounded waits run out: the kernels record MQ_DEV_TIMEOUT in the
 * device status word, write no output and return; the GPU context stays
 * usable.  MQ_FAULT_WITHHOLD_RECORDS: in the persistent step kernel the last
 * CTA (which always owns h blocks) never writes its h records and every wait is limited to 50 ms, so every
 * CTA's down phase runs out of time waiting for them: the kernel records
 * MQ_DEV_TIMEOUT, the abort word stops every CTA, and the launch returns.
 * MQ_FAULT_WITHHOLD_COUNT: in the persistent step kernel the last CTA never
 * adds its finished phases to the phase counter (waits limited to 50 ms), so
 * every CTA's wait for the first phase's end runs out, with the same outcome.
 * MQ_FAULT_NONE restores normal operation. */
#define MQ_FAULT_NONE 0
#define MQ_FAULT_WITHHOLD_TILE 1
#define MQ_FAULT_WITHHOLD_RECORDS 2
#define MQ_FAULT_WITHHOLD_COUNT 3
mq_status mq_debug_set_fault(int32_t fault);

/* Test-only view of the launch planner, on the host: no GPU and no mq_init
 * needed.  Gives the plan a call would take on a device with num_sms SMs,
 * l2_bytes of L2 and max_smem bytes of opt-in shared memory per block, under
 * the current variant policy.
 *  - mq_debug_plan_mv: one q4_K projection as mq_matvec_q4K_q8_0
 *    (MQ_PLAN_MATVEC: rows x K) or mq_ffn_gu_silu_down plans it
 *    (MQ_PLAN_GATE_UP: rows = 2I, K = H, I given; MQ_PLAN_DOWN: rows = H,
 *    K = I).  Writes MQ_PLAN_FIELDS values to out.
 *  - mq_debug_plan_step: the persistent step (MQ_STEP_PERSISTENT) of *shape.
 *    Writes MQ_STEP_PLAN_FIELDS values, then MQ_PLAN_FIELDS values for each
 *    phase (qkv, o, gate/up, down; a phase left out has variant 0 and rows
 *    per CTA 0).
 * Per-projection fields, in order: 0 variant (1: bulk-copy ring kernels,
 * 0: register-streaming kernels), 1 grid, 2 block, 3 dynamic shared memory
 * bytes, 4 C (ring plans: 128-weight units per row or per part of a K split;
 * register plans: 64-weight chunks), 5 L (lanes per item), 6 S (units, or
 * half-units, per segment), 7 nseg (segments per row), 8 consumer warps,
 * 9 row-lanes per segment, 10 T (rows per tile), 11 ring stages, 12 bytes
 * per stage, 13 rows per CTA, 14 column lanes (0/1), 15 warps per column
 * group (0: none), 16 warps with work per group, 17 half-unit lanes (0/1),
 * 18 K-split parts (1: whole rows), 19 super-blocks per part (0: whole rows).
 * Step fields: 0 grid, 1 block, 2 dynamic shared memory bytes, 3 consumer
 * warps, 4 ring stages, 5 bytes per stage, 6 L2-prefetched tiles per CTA,
 * 7 workspace bytes.
 * Both return MQ_ERR_INVALID_ARG for a null pointer, an n_out smaller than
 * what they write, a bad kind or a non-positive device description; the
 * shape checks of the call they stand for (MQ_ERR_SHAPE ...); and
 * MQ_ERR_UNSUPPORTED where that call would find no plan on the device.
 * Nothing is written unless they return MQ_OK. */
#define MQ_PLAN_MATVEC 0
#define MQ_PLAN_DOWN 1
#define MQ_PLAN_GATE_UP 2
#define MQ_PLAN_FIELDS 20
#define MQ_STEP_PLAN_FIELDS 8
mq_status mq_debug_plan_mv(int32_t kind, int64_t rows, int32_t K, int32_t ncols, int32_t I, int32_t num_sms,
                           int64_t l2_bytes, int32_t max_smem, int64_t* out, int32_t n_out);
mq_status mq_debug_plan_step(const mq_step_shape* shape, int32_t num_sms, int64_t l2_bytes, int32_t max_smem,
                             int64_t* out, int32_t n_out);

#ifdef __cplusplus
}
#endif

#endif /* MQ_H */
