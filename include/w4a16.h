/*
 * w4a16.h -- C ABI of libw4a16.so: INT4 weight / float activation GEMMs with symmetric
 * group-32 quantization, for NVIDIA GB300 (sm_103a).
 *
 * Weight format (page "The Weight of Precision: Building Native INT4 Quantization for a Custom
 * Speculative Decoding Engine", section "The Kernel: w4a16_gemm"; page "The First Line of Code:
 * Implementing W4A16 Quantization in a Native Speculative Decoding Engine", section "What the
 * Edit Actually Does"):
 *   - a weight matrix W[K, N] maps K inputs to N outputs;
 *   - codes are 4-bit, value = nibble - 8, range [-8, 7];
 *   - qw[K/8, N] int32, row-major: word (i, n) holds k = 8i .. 8i+7 of column n, code 8i+j in
 *     bits [4j, 4j+3] (lowest nibble = lowest k);
 *   - sc[K/32, N] float32, row-major: one scale per group of 32 consecutive k per column n;
 *   - dequantized weight w[k, n] = (nibble - 8) * sc[k/32, n].
 *
 * Conventions for every entry point below:
 *   - all tensor pointers are DEVICE pointers (cudaMalloc or a caching allocator), row-major,
 *     owned by the caller; the library never allocates device memory, never frees, and never
 *     synchronizes the stream (except where an entry says so);
 *   - tensor pointers must be 16-byte aligned, else W4A16_ERR_ALIGN;
 *   - `group` must be 32 (W4A16_GROUP), else W4A16_ERR_UNSUPPORTED;
 *   - K must be a positive multiple of 32; N a multiple of 4 (8 for bf16 outputs), else
 *     W4A16_ERR_ARG; M = 0 or N = 0 is an empty call and returns W4A16_OK without launching;
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); work is asynchronous on it;
 *   - arguments are checked before anything is launched; a failed check launches nothing;
 *   - a launch failure returns W4A16_ERR_CUDA (the CUDA error is kept for
 *     w4a16_last_cuda_error());
 *   - outputs may not alias inputs.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_GROUP 32
#define W4A16_ABI_VERSION 1

/* Same type as cudaStream_t. */
typedef struct CUstream_st* w4a16_stream_t;

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_ARG = 1,          /* a size or pointer argument is invalid */
  W4A16_ERR_ALIGN = 2,        /* a tensor pointer is not 16-byte aligned */
  W4A16_ERR_UNSUPPORTED = 3,  /* valid but unsupported (group != 32, no sm_103 device, ...) */
  W4A16_ERR_WORKSPACE = 4,    /* workspace missing or smaller than the size query returns */
  W4A16_ERR_CUDA = 5,         /* a CUDA call or kernel launch failed */
  W4A16_ERR_NOT_FOUND = 6,    /* linear(): no quantized weight registered under that name */
  W4A16_ERR_IO = 7,           /* loader: file missing, unreadable or of the wrong size */
  W4A16_ERR_TIMEOUT = 8       /* a kernel gave up a bounded wait (see w4a16_device_error) */
} w4a16_status;

/* Human-readable name of a status code (static string). */
const char* w4a16_status_string(w4a16_status s);
/* W4A16_ABI_VERSION of the loaded library. */
int w4a16_abi_version(void);
/* The CUDA error code (cudaError_t as int) behind the last W4A16_ERR_CUDA of this thread. */
int w4a16_last_cuda_error(void);

/* ------------------------------------------------------------------------------------------
 * Quantize + pack (offline step). Page "The Weight of Precision ...", sections "The Kernel:
 * w4a16_gemm" and "The Reference and Bundle Pipeline" (.qw int32 and .sc float32 arrays).
 *   W   [K, N] float32 in;  qw [K/8, N] int32 out;  sc [K/32, N] float32 out.
 *   s = max_{k in group} |W[k,n]| / 7 (float32),  q = clamp(rint(W / s), -8, 7) with the
 *   float32 quotient rounded half to even; an all-zero group gives s = 0 and q = 0.
 * Results are bit-identical to the reference quantizer for finite inputs. */
w4a16_status w4a16_quantize(const float* W, int K, int N, int group,
                            int32_t* qw, float* sc, w4a16_stream_t stream);

/* Unpack + dequantize: W[k, n] = (nibble - 8) * sc[k/32, n] rounded to float32.
 * Page "The First Line of Code ...", section "What the Edit Actually Does" (dequantization
 * must be identical between the reference and the kernel). */
w4a16_status w4a16_dequantize(const int32_t* qw, const float* sc, int K, int N, int group,
                              float* W, w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * y[M, N] = x[M, K] @ dequant(qw, sc), float32 activations and output, float32 accumulation.
 * Page "The Final Wire: How a Single Edit Integrated INT4 Quantization into a Native DDTree
 * Inference Engine", section "The Multi-Step Integration Chain", step 1; page "The Weight of
 * Precision ...", section "The Kernel: w4a16_gemm".
 * Any M >= 0; the kernels are built for the decode / draft-tree-verify regime (M <= 16):
 * larger M runs as 16-row slices within one launch, the slices of a weight tile resident
 * together so each weight byte comes from HBM once per call. Deterministic (fixed reduction
 * order). */
w4a16_status w4a16_gemm(const float* x, const int32_t* qw, const float* sc, float* y,
                        int M, int N, int K, int group, w4a16_stream_t stream);

/* Fused gate/up projection of a SwiGLU MLP with the activation in the epilogue:
 *   h = x[M, K] @ dequant(qw_gu, sc_gu)   with qw_gu [K/8, N2], gate = columns [0, N2/2),
 *                                          up = columns [N2/2, N2)
 *   y[M, N2/2] = silu(gate) * up,  silu(z) = z / (1 + exp(-z)).
 * x is read once for both halves. Page "The Final Wire ...", section "What the Edit Actually
 * Changes" (MLP gate, up and down projections); N2 must be a multiple of 8. */
w4a16_status w4a16_gemm_swiglu(const float* x, const int32_t* qw_gu, const float* sc_gu,
                               float* y, int M, int N2, int K, int group,
                               w4a16_stream_t stream);

/* GEMM with bf16 activations x[M, K] (bit patterns) and bf16 output y[M, N], float32
 * accumulation. M > 16 (prefill) runs the tensor-core contraction with the dequantized weights
 * rounded to bf16; M <= 16 runs the weight-streaming kernels in bf16 form (exact codes, scale
 * applied in float32 per group). Not on the pages (their activations are float32); tolerance
 * 1e-2 relative L2 against the exact product. Needs an sm_103 device; K % 64 == 0, N % 8 == 0,
 * x and y 16-byte aligned. Deterministic. */
w4a16_status w4a16_gemm_bf16(const uint16_t* x, const int32_t* qw, const float* sc,
                             uint16_t* y, int M, int N, int K, int group,
                             w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Routed-expert MoE block (page "The Final Wire ...", section "What the Edit Actually Changes":
 * per token the router picks top-k experts; each expert's gate, up and down projections run
 * through the INT4 GEMM):
 *   out[t, :] = sum_{j < topk} topk_w[t, j] * down_e( silu(g) * u ),  (g | u) = x[t] @ W_gu[e],
 *   e = topk_ids[t, j].
 *   x        [T, K] float32          topk_ids [T, topk] int32 in [0, E)    topk_w [T, topk] f32
 *   qw_gu    [E, K/8, 2I] int32      sc_gu    [E, K/32, 2I] float32   (gate | up per expert)
 *   qw_dn    [E, I/8, K]  int32      sc_dn    [E, I/32, K]  float32
 *   out      [T, K] float32 (overwritten)
 * Every expert's weights are read once per call, whatever number of tokens it received.
 * `workspace` is device memory of at least w4a16_moe_workspace_size(T, topk, E, K, I) bytes,
 * 16-byte aligned; its contents need no initialisation and are scratch after the call.
 * Expert ids outside [0, E) are not checked on the host (the ids live on the device); the
 * routing kernel skips such pairs and flags W4A16_ERR_ARG in the device error word.
 * K and I must be multiples of 32; I a multiple of 8. Deterministic. */
size_t w4a16_moe_workspace_size(int T, int topk, int E, int K, int I);
w4a16_status w4a16_moe_gemm(const float* x, const int32_t* topk_ids, const float* topk_w,
                            int T, int topk, int E,
                            const int32_t* qw_gu, const float* sc_gu,
                            const int32_t* qw_dn, const float* sc_dn,
                            float* out, int K, int I, int group,
                            void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* MoE block with a shared expert (page "The Weight of Precision ...", section "The Engine
 * Dispatch: Model::linear": the MoE experts, the shared expert and the dense MLP layers run
 * through the INT4 path):
 *   out[t, :] = down_s( silu(g_s) * u_s ) + sum_{j < topk} topk_w[t, j] * down_e(...),
 *   (g_s | u_s) = x[t] @ W_gu_shared,
 * i.e. w4a16_moe_gemm plus one expert that every token goes through with weight 1.
 *   qs_gu [K/8, 2 Is] int32, ss_gu [K/32, 2 Is] float32   (gate | up of the shared expert)
 *   qs_dn [Is/8, K] int32,   ss_dn [Is/32, K] float32
 * Other arguments as w4a16_moe_gemm; Is a multiple of 32; the shared expert's weights 16-byte
 * aligned. `workspace` holds at least w4a16_moe_block_workspace_size(T, topk, E, K, I, Is) bytes.
 * The shared expert runs as two dense small-M GEMMs (16-row slices in one launch each); its output
 * seeds each row of the combine, which then adds the routed rows in slot order. Deterministic. */
size_t w4a16_moe_block_workspace_size(int T, int topk, int E, int K, int I, int Is);
w4a16_status w4a16_moe_block(const float* x, const int32_t* topk_ids, const float* topk_w,
                             int T, int topk, int E,
                             const int32_t* qw_gu, const float* sc_gu,
                             const int32_t* qw_dn, const float* sc_dn,
                             const int32_t* qs_gu, const float* ss_gu,
                             const int32_t* qs_dn, const float* ss_dn, int Is,
                             float* out, int K, int I, int group,
                             void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* The same MoE block for callers that cannot allocate device memory, such as a plugin or
 * foreign-function interface that only passes input and output buffers, or a process whose
 * device memory another runtime has already reserved. The pages have no counterpart: this is
 * an addition of this library.
 *   - Arguments and results as w4a16_moe_gemm, without the workspace: the scratch is one array
 *     of W4A16_MOE_STATIC_SCRATCH_BYTES in device memory that the library's device code holds on
 *     every GPU that loads it, until the process exits or the device is reset. No allocation
 *     happens in the call.
 *   - The argument checks and their order are those of w4a16_moe_gemm; then sizes with
 *     w4a16_moe_workspace_size(T, topk, E, K, I) > W4A16_MOE_STATIC_SCRATCH_BYTES are refused
 *     with W4A16_ERR_WORKSPACE before anything is launched (at K = 7168, I = 2048 that allows
 *     up to 909 token-expert pairs for any E <= 4096, e.g. T = 64 tokens with top-8).
 *   - Each call outside stream capture looks up the array's device address (with the device
 *     current), so a device reset, which releases the array, does not leave a stale address.
 *     A call under stream capture reuses the last address looked up on that device: make one
 *     call on the device before capturing (else W4A16_ERR_CUDA).
 *   - All calls on a device share the one array and it keeps whatever the last call left there
 *     (nothing in it needs to start at zero). Calls whose execution overlaps on the GPU -- on
 *     different streams, or from different host threads -- race on it; serialize them. */
#define W4A16_MOE_STATIC_SCRATCH_BYTES (32u << 20)
w4a16_status w4a16_moe_gemm_noalloc(const float* x, const int32_t* topk_ids,
                                    const float* topk_w, int T, int topk, int E,
                                    const int32_t* qw_gu, const float* sc_gu,
                                    const int32_t* qw_dn, const float* sc_dn,
                                    float* out, int K, int I, int group,
                                    w4a16_stream_t stream);

/* Router weights over each token's selected experts: weights[t, :] = softmax(logits[t, :]).
 * logits, weights: [T, topk] float32, 1 <= topk <= 32. */
w4a16_status w4a16_topk_softmax(const float* logits, float* weights, int T, int topk,
                                w4a16_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Loader: raw little-endian .qw (int32 [K/8, N]) and .sc (float32 [K/32, N]) files into
 * caller-owned device buffers (page "The Final Wire ...", section "The Multi-Step Integration
 * Chain", steps 3 and 5). Uses a host staging buffer it allocates and frees itself; copies
 * synchronously. W4A16_ERR_IO if a file is missing or its size is not exactly the expected
 * byte count. */
w4a16_status w4a16_load_qw_sc(const char* qw_path, const char* sc_path, int K, int N,
                              int group, int32_t* qw, float* sc);

/* ------------------------------------------------------------------------------------------
 * Name -> quantized weight registry and linear() dispatch (page "The Final Wire ...", section
 * "What the Edit Actually Changes"; page "The Weight of Precision ...", section "The Engine
 * Dispatch: Model::linear"). Unlike the pages' dispatcher there is NO silent float fallback:
 * a name that was never registered returns W4A16_ERR_NOT_FOUND (the pages flag the silent
 * fallback as a correctness risk, "Assumptions in the Design", assumptions 1 and 3).
 * The registry stores device pointers it does not own. Host memory only; not thread-safe
 * for concurrent add/destroy. */
typedef struct w4a16_registry w4a16_registry;
w4a16_registry* w4a16_registry_create(void);
void w4a16_registry_destroy(w4a16_registry* reg);
/* Registers (or replaces) `name`. Pointers are checked for alignment; K, N, group as above. */
w4a16_status w4a16_registry_add(w4a16_registry* reg, const char* name, const int32_t* qw,
                                const float* sc, int K, int N, int group);
/* Looks `name` up; K and N (either may be NULL) receive its shape. */
w4a16_status w4a16_registry_find(const w4a16_registry* reg, const char* name, int* K, int* N);
/* y[M, N] = x[M, K] @ W_name  (dispatches to w4a16_gemm). */
w4a16_status w4a16_linear(const w4a16_registry* reg, const char* name, const float* x,
                          float* y, int M, w4a16_stream_t stream);
/* y[M, N/2] = silu(gate) * up with W_name = [gate | up]  (dispatches to w4a16_gemm_swiglu). */
w4a16_status w4a16_linear_swiglu(const w4a16_registry* reg, const char* name, const float* x,
                                 float* y, int M, w4a16_stream_t stream);

/* Multi-tensor weight bundle (page "The Final Wire ...", section "The Multi-Step Integration
 * Chain", steps 3 and 5: a generator writes bundles of quantized weights and scales; the engine
 * maps weight names to them). The pages give no byte layout; this library's is, little-endian:
 *   "W4A16BDL" (8 bytes), u32 version = 1, u32 count,
 *   count x { u32 name_len, name (no terminator), i32 K, i32 N, u64 qw_offset, u64 sc_offset },
 *   then the blobs qw [K/8, N] int32 and sc [K/32, N] float32 at their file offsets.
 * Names are unique, K a multiple of 32, N of 4. w4a16_bundle_info reads the index only and
 * reports the number of tensors and the device bytes w4a16_bundle_load needs. w4a16_bundle_load
 * copies every tensor into `arena` (caller-owned device memory, 256-byte aligned, each blob at
 * a 256-byte boundary), synchronously, and adds each name to `reg`, which then points into the
 * arena. W4A16_ERR_IO for an unreadable or malformed file (nothing is copied for a malformed
 * index), W4A16_ERR_WORKSPACE for a too small arena. The Python writer is
 * int4_w4a16_group_gb300/bundle.py. */
w4a16_status w4a16_bundle_info(const char* path, int* count, size_t* device_bytes);
w4a16_status w4a16_bundle_load(w4a16_registry* reg, const char* path, void* arena,
                               size_t arena_bytes);

/* ------------------------------------------------------------------------------------------
 * Device error word. Kernels that wait on a barrier give up after a bounded number of polls
 * and record a status here instead of hanging. Synchronizes the device, returns the recorded
 * status in *code (W4A16_OK if none) and clears it. */
w4a16_status w4a16_device_error(int* code);

/* Self-test of that path: one thread waits on a shared-memory barrier with the kernels' own
 * polled, time-limited wait. arrive = 0: nothing arrives, the wait gives up after limit_us
 * microseconds (1 .. 100000, else W4A16_ERR_ARG) and records W4A16_ERR_TIMEOUT in the device
 * error word; arrive = 1: the thread arrives first and nothing is recorded. Asynchronous on
 * `stream`; read the outcome with w4a16_device_error. */
w4a16_status w4a16_selftest_wait(int arrive, int limit_us, w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* W4A16_H_ */
