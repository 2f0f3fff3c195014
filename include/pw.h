/*
 * pw.h -- C ABI of the PagedWeight fused mixed-precision MoE layer (libpw.so).
 *
 * The layer is the one described on the PagedWeight pages:
 *   - "Core components" 1, Paged Weight representation: experts' weights are
 *     stored per linear block (layer, expert, module in {gate_up, down}) in
 *     Any-Precision's overlay bitplane format with lookup tables (LUTs); a
 *     Weight Page Table tracks each block's committed bitwidth q_i and its page
 *     state (GPU-resident, CPU-resident or in transfer).
 *   - "Core components" 3, asynchronous execution and kernel optimisation: a
 *     fused mixed-precision kernel reads the bitplanes and LUTs directly and
 *     supports a different bitwidth per linear block inside one fused
 *     operation; bitwidth commits only take effect at safe boundaries so that
 *     inference is never interrupted.
 *
 * Storage format (the pages give none; this is the library's contract):
 *   - A block with N rows and K columns (K % 32 == 0) stores 8 bitplanes of
 *     its 8-bit codes, uint32 [8][K/32][N], plane-major.  Plane p holds bit
 *     (7 - p) of every code (plane 0 = most significant), so the top q planes
 *     are the first q planes, a contiguous prefix.  Within a plane, word w of
 *     row n (at [p][w][n]) holds columns 32w..32w+31 of row n, column 32w+t
 *     at bit t; the N words of a word column are contiguous, so 32
 *     consecutive rows' words are 128 contiguous bytes.
 *   - Reading q planes gives idx_q = code >> (8 - q).  Row n's q-bit LUT holds
 *     2^q fp16 values, fp16 [N][2^q]; the weight is LUT_q[n][idx_q].
 *   - Expert e owns block 2e (gate_up, N = 2I rows x K = H: rows 0..I-1 gate,
 *     rows I..2I-1 up) and block 2e+1 (down, N = H rows x K = I).
 *   - Supported committed bitwidths: q in {3, 4, 5, 6, 8}.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be device memory (or managed
 *     memory) of the current device; they stay owned by the caller.  Host
 *     pointers are read before the call returns.
 *   - Work is enqueued on `stream` and is asynchronous; nothing synchronises
 *     the host unless the comment says so.
 *   - The return value is a status code (PW_OK = 0).  On failure nothing is
 *     enqueued and pw_last_error() returns a message (thread-local).  No C++
 *     exception crosses the ABI.
 *   - Errors found on the device (an expert id out of range, a page that is
 *     not GPU-resident) never trap: the offending unit of work is skipped and
 *     the first such code is latched in the page table's status word, read
 *     with pw_page_table_status().  Every device-side wait of the forward
 *     kernels (mbarrier waits in the tcgen05 kernels, the decode down
 *     kernel's wait for an expert's gate_up tiles) is bounded; one that runs
 *     out latches PW_ERR_TIMEOUT and the kernel returns.
 */
#ifndef PW_H_
#define PW_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define PW_OK                     0
#define PW_ERR_INVALID_ARG        1  /* null pointer, negative size, bad enum        */
#define PW_ERR_UNSUPPORTED_Q      2  /* q not in {3,4,5,6,8} (or b not in 1..8)      */
#define PW_ERR_SHAPE              3  /* K % 32 != 0, table size != 2E, size limits   */
#define PW_ERR_WORKSPACE          4  /* workspace null or smaller than required      */
#define PW_ERR_PAGE_NOT_RESIDENT  5  /* device: a routed block is not GPU-resident   */
#define PW_ERR_BAD_EXPERT_ID      6  /* device: topk id outside [0, E)               */
#define PW_ERR_CUDA               7  /* a CUDA runtime call failed                   */
#define PW_ERR_TIMEOUT            8  /* a bounded device wait gave up                */
#define PW_ERR_UNSUPPORTED_DEVICE 9  /* the current device is not sm_103             */
#define PW_ERR_RANGE             10  /* device: a LUT value outside the range a block
                                        committed at q <= 4 supports (|v| >= 2048 or
                                        not finite); the block is still computed      */
#define PW_ERR_NOT_BUILT         11  /* this library was built without the facility  */

/* ---- page states of the Weight Page Table ------------------------------ */
#define PW_PAGE_GPU          0  /* planes and LUT are in device memory        */
#define PW_PAGE_CPU          1  /* offloaded to host memory: not readable     */
#define PW_PAGE_IN_TRANSFER  2  /* a copy is in flight: not readable          */

/* ---- forward paths ----------------------------------------------------- */
#define PW_PATH_AUTO     0  /* decode kernels for small token counts, else prefill */
#define PW_PATH_DECODE   1  /* CUDA-core fused decode kernels; within a call of
                                >= 16 tokens, experts holding >= 8 pairs go
                                through the tcgen05 GEMM kernels (when the shape
                                allows them)                                        */
#define PW_PATH_PREFILL  2  /* dequantise-to-shared-memory tcgen05 GEMM kernels     */

/* One linear block's page-table entry (24 bytes).  PagedWeight, "Core
 * components" 1: the Weight Page Table keeps each block's committed bitwidth
 * q_i and page state; this entry adds where the block's planes and its
 * committed LUT live. */
typedef struct pw_block_entry {
  int32_t q;               /* committed bitwidth q_i, in {3,4,5,6,8}                   */
  int32_t state;           /* PW_PAGE_*                                                */
  const uint32_t* planes;  /* device: uint32 [>= q][K/32][N], the block's planes      */
  const uint16_t* lut;     /* device: fp16 [N][2^q], the LUT for the committed q       */
} pw_block_entry;

/* Shape of one routed-expert layer call. */
typedef struct pw_moe_shape {
  int32_t T;  /* tokens (>= 0)                                  */
  int32_t H;  /* hidden size (> 0, multiple of 32)               */
  int32_t I;  /* expert intermediate size (> 0, multiple of 32)  */
  int32_t E;  /* experts (> 0); the page table holds 2E blocks   */
  int32_t k;  /* experts per token (1..E)                        */
} pw_moe_shape;

/* Opaque Weight Page Table.  Its entry array sits at one fixed device
 * address for the table's lifetime, so a CUDA graph that captured a forward
 * call keeps reading the current commits. */
typedef struct pw_page_table pw_page_table;

/* Last error message of the calling thread ("" if none). */
const char* pw_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pw_version(void);

/* ---- bitplane encoding -------------------------------------------------
 * Encode 8-bit codes into the overlay bitplane format (PagedWeight, "Core
 * components" 1, APL overlay bitplanes).
 *   codes  device uint8 [N][K], row-major
 *   planes device uint32 [8][K/32][N] (output)
 * Errors: PW_ERR_INVALID_ARG (null, N < 0), PW_ERR_SHAPE (K % 32 != 0 or
 * K <= 0). */
int pw_pack_bitplanes(const uint8_t* codes, int32_t N, int32_t K,
                      uint32_t* planes, cudaStream_t stream);

/* Read a block's top b planes back into b-bit indices, idx = code >> (8-b)
 * (PagedWeight, "Core components" 1: a b-bit view reads the top b planes).
 * Exposed so that the bit extraction can be checked bit-exactly.
 *   planes device uint32 [>= b][K/32][N];  idx device uint8 [N][K] (output)
 * Errors: PW_ERR_INVALID_ARG, PW_ERR_SHAPE, PW_ERR_UNSUPPORTED_Q (b not in 1..8). */
int pw_unpack_top(const uint32_t* planes, int32_t N, int32_t K, int32_t b,
                  uint8_t* idx, cudaStream_t stream);

/* ---- routing -------------------------------------------------------------
 * Router: softmax over E logits, top-k experts (ties to the lower id), the k
 * kept probabilities renormalised to sum to 1.  The pages describe routing
 * only through the routing mass the planner tracks (PagedWeight, "Core
 * components" 2, online routing statistics); the layer itself consumes its
 * output.
 *   logits       device float [T][E]
 *   topk_ids     device int32 [T][k]  (output, descending probability)
 *   topk_weights device float [T][k]  (output)
 * Limits: 1 <= k <= E <= 1024 and k <= 32.  Errors: PW_ERR_INVALID_ARG, PW_ERR_SHAPE. */
int pw_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                  int32_t* topk_ids, float* topk_weights, cudaStream_t stream);

/* Token-to-expert permutation (the dispatch step of the fused layer,
 * PagedWeight "Core components" 3).  Pair p = t*k + j goes to expert
 * topk_ids[t][j]; pairs are grouped by expert, ascending p inside an expert.
 *   topk_ids device int32 [T][k]
 *   offsets  device int32 [E+1] (output): expert e owns perm[offsets[e] .. offsets[e+1])
 *   perm     device int32 [T*k] (output): pair ids in grouped order
 *   inv      device int32 [T*k] (output, may be NULL): inv[perm[r]] = r
 * Limits: E <= 1024.  An id outside [0, E) latches PW_ERR_BAD_EXPERT_ID in
 * *status_out (device int32, may be NULL) and that pair is dropped (it then
 * appears in no expert's range and its inv entry is -1). */
int pw_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
               int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* status_out,
               cudaStream_t stream);

/* ---- Weight Page Table ----------------------------------------------------
 * PagedWeight, "Core components" 1 (Weight Page Table: committed bitwidth q_i
 * and page state per linear block) and 3 (bitwidth commits applied only at a
 * safe boundary).
 *
 * Create a table of num_blocks entries from host_init (host array).  Allocates
 * device memory and synchronises the current device once.  Errors:
 * PW_ERR_INVALID_ARG, PW_ERR_UNSUPPORTED_Q, PW_ERR_CUDA. */
int pw_page_table_create(int32_t num_blocks, const pw_block_entry* host_init,
                         pw_page_table** out);

/* Free a table (synchronises the device first).  NULL is accepted. */
int pw_page_table_destroy(pw_page_table* table);

/* Recommit: for i < n, block block_ids[i] takes bitwidth new_q[i] and reads
 * the LUT at new_lut[i] (a device pointer to fp16 [N][2^new_q]).  The update
 * is a kernel enqueued on `stream` (host arrays are passed by value), so a
 * forward call enqueued later on the same stream sees the new bitwidths and
 * one enqueued earlier sees the old ones: the stream order is the safe
 * boundary.  The planes pointer is unchanged: lowering q only stops reading
 * the tail planes.  Errors: PW_ERR_INVALID_ARG (n < 0, id out of range, null
 * lut), PW_ERR_UNSUPPORTED_Q. */
int pw_page_table_commit(pw_page_table* table, int32_t n, const int32_t* block_ids,
                         const int32_t* new_q, const uint16_t* const* new_lut,
                         cudaStream_t stream);

/* Move pages: for i < n, block block_ids[i] reads its planes from planes[i]
 * (device pointer) and takes page state states[i] (PW_PAGE_*).  Stream-ordered
 * like pw_page_table_commit.  A forward call skips every routed block whose
 * state is not PW_PAGE_GPU and latches PW_ERR_PAGE_NOT_RESIDENT. */
int pw_page_table_set_pages(pw_page_table* table, int32_t n, const int32_t* block_ids,
                            const uint32_t* const* planes, const int32_t* states,
                            cudaStream_t stream);

/* Copy the current entries to host_out[num_blocks] (host).  Synchronises `stream`. */
int pw_page_table_read(const pw_page_table* table, pw_block_entry* host_out,
                       cudaStream_t stream);

/* Number of entries. */
int32_t pw_page_table_size(const pw_page_table* table);

/* Read the device status word latched by forward calls into *host_status
 * (PW_OK or the first device-side error) and clear it if reset != 0.
 * Synchronises `stream`. */
int pw_page_table_status(pw_page_table* table, int32_t* host_status, int32_t reset,
                         cudaStream_t stream);

/* Online routing statistics (PagedWeight, "Core components" 2: the planner
 * tracks each expert's routing mass, its selection frequency and weight).
 * While set, every forward call through `table` adds, for each expert e,
 *   counts[e] += number of (token, j) pairs routed to e,
 *   mass[e]   += sum of their topk_weights,
 * as a by-product of grouping the pairs (pairs with an id outside [0, E) are
 * left out).  counts: device int32 [E]; mass: device float [E]; both owned and
 * zeroed by the caller, who reads them back (e.g. to derive hot experts for the
 * planner).  Pass NULL, NULL to stop.  The float sums are accumulated with
 * atomics, so their last bits depend on the order of the additions.
 * Errors: PW_ERR_INVALID_ARG (NULL table, exactly one buffer NULL). */
int pw_page_table_set_routing_stats(pw_page_table* table, int32_t* counts, float* mass);

/* ---- page movement ---------------------------------------------------------
 * PagedWeight, "Core components" 3: weight pages are offloaded to CPU RAM and
 * reloaded asynchronously to hide the latency; a bitwidth commit takes effect
 * only at a safe boundary.  Planes are plane-major ([8][K/32][N]), so the tail
 * planes p >= q of a block, which a forward call at bitwidth q never reads,
 * are one contiguous run: lowering q frees them, raising q needs them back.
 *
 * Copy planes [p_begin, 8) of a block (device, N rows, K columns) to pinned
 * host memory, or back, on `stream` (asynchronous; one cudaMemcpyAsync).
 * host: (8 - p_begin) * N * K / 8 bytes.  Errors: PW_ERR_INVALID_ARG (NULL,
 * unaligned planes, p_begin outside 0..7, N < 0), PW_ERR_SHAPE (K % 32),
 * PW_ERR_CUDA. */
int pw_planes_to_host(const uint32_t* planes, int32_t N, int32_t K, int32_t p_begin, void* host,
                      cudaStream_t stream);
int pw_planes_from_host(const void* host, uint32_t* planes, int32_t N, int32_t K, int32_t p_begin,
                        cudaStream_t stream);

/* pw_page_table_commit ordered after `ready` (e.g. an event recorded on the
 * copy stream after pw_planes_from_host): `stream` waits for the event, then
 * commits, so forward calls enqueued on `stream` before this call read the old
 * bitwidths and calls after it the new ones, never a half-copied tail.
 * Errors: as pw_page_table_commit, plus PW_ERR_CUDA. */
int pw_page_table_commit_after(pw_page_table* table, int32_t n, const int32_t* block_ids,
                               const int32_t* new_q, const uint16_t* const* new_lut,
                               cudaEvent_t ready, cudaStream_t stream);

/* ---- planner ----------------------------------------------------------------
 * Greedy damage-per-byte planner (PagedWeight, "Core components" 2: when a
 * memory target is set, the planner scores the damage of each possible
 * bitwidth cut and greedily takes the cuts with the least damage per byte
 * saved; frequently routed experts are protected by higher bitwidth floors
 * and damage multipliers).  Host-only computation; its output is the list a
 * pw_page_table_commit applies.
 *   n_blocks       2E blocks, block 2e = gate_up and 2e+1 = down of expert e
 *   q_now          host int32 [n_blocks], current bitwidths (3,4,5,6,8)
 *   sensitivity    host float [n_blocks], damage per unit of quantisation error (>= 0)
 *   bytes_per_bit  host int64 [n_blocks], bytes of one bitplane of the block (N*K/8)
 *   routing_mass   host float [E], each expert's routing mass (>= 0), e.g. the
 *                  mass accumulated by pw_page_table_set_routing_stats
 *   hot_floor      bitwidth floor of hot experts (3,4,5,6,8); an expert is hot
 *                  when its share of the total mass exceeds 1/E; others: floor 3
 *   bytes_to_free  the memory target
 * A cut lowers one block by one rung of 8 > 6 > 5 > 4 > 3, from b to b', and
 *   damage = sensitivity * m_e * (4^-b' - 4^-b),  m_e = max(1, E * share_e),
 *   bytes  = (b - b') * bytes_per_bit
 * (4^-b: the relative error of a b-bit quantiser).  The planner repeatedly
 * applies the cut with the least damage per byte (ties: lower block id) until
 * at least bytes_to_free bytes are saved or no cut is left.
 * Outputs: out_ids / out_q (host int32 [n_blocks]) = the blocks whose bitwidth
 * changed, ascending id, and their new bitwidth; *n_out their number;
 * *bytes_freed the bytes the cuts save.
 * Errors: PW_ERR_INVALID_ARG (NULL pointer, n_blocks odd or negative, negative
 * input), PW_ERR_UNSUPPORTED_Q (a bitwidth off the ladder). */
int pw_plan_recommit(int32_t n_blocks, const int32_t* q_now, const float* sensitivity,
                     const int64_t* bytes_per_bit, const float* routing_mass, int32_t hot_floor,
                     int64_t bytes_to_free, int32_t* out_ids, int32_t* out_q, int32_t* n_out,
                     int64_t* bytes_freed);

/* ---- the fused layer ------------------------------------------------------
 * Bytes of device workspace a forward call of this shape needs. */
int pw_workspace_bytes(const pw_moe_shape* shape, size_t* bytes);

/* The fused mixed-precision MoE expert layer (PagedWeight, "Core components"
 * 3): for every token t,
 *   out[t] = sum_j topk_weights[t][j] * y_{e}(x_t),   e = topk_ids[t][j],
 *   y_e(x) = (SiLU(x W_gate,e^T) * (x W_up,e^T)) W_down,e^T,
 * where every weight is LUT_q[n][code >> (8-q)] read from the block's top q
 * bitplanes at the q committed in `table` when the call runs on the stream.
 *   hidden       device bf16 [T][H] (raw bits), row-major
 *   topk_ids     device int32 [T][k]
 *   topk_weights device float [T][k]
 *   table        page table with 2E entries
 *   out          device float [T][H] (output, overwritten)
 *   workspace    device scratch of >= pw_workspace_bytes(shape) bytes, 256-byte
 *                aligned; it must not be in use by another call in flight
 * hidden, topk_ids, topk_weights and out may also be pinned host memory that
 * the device addresses with the same pointer (cudaHostAlloc or
 * cudaHostRegister under unified addressing): the kernels then read the
 * inputs and write the output across the CPU-GPU link themselves, so a step
 * needs no separate copies.
 * The call allocates nothing and never synchronises the host; it can be
 * captured in a CUDA graph.  Errors: PW_ERR_INVALID_ARG, PW_ERR_SHAPE,
 * PW_ERR_WORKSPACE, PW_ERR_UNSUPPORTED_DEVICE, PW_ERR_CUDA. */
int pw_moe_forward(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                   const float* topk_weights, const pw_page_table* table, float* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* pw_moe_forward with an explicit path (PW_PATH_*); PW_PATH_AUTO is what
 * pw_moe_forward uses.  Both paths compute the same function. */
int pw_moe_forward_path(const pw_moe_shape* shape, const void* hidden, const int32_t* topk_ids,
                        const float* topk_weights, const pw_page_table* table, float* out,
                        void* workspace, size_t workspace_bytes, int32_t path,
                        cudaStream_t stream);

/* The fused layer fed with router logits (PagedWeight, "Core components" 3:
 * one fused operation; "Core components" 2: the routing mass the planner
 * tracks is these weights).  The routing, softmax over the E logits, the top
 * k experts (ties to the lower id) and the kept probabilities renormalised,
 * runs inside the launch that groups the pairs (the decode path's prep, the
 * prefill path's permutation), so the call needs no separate router launch;
 * its result is written to topk_ids / topk_weights (caller-owned outputs,
 * also the ids and weights the layer then uses), as pw_route_topk would write
 * it.  Otherwise the same as pw_moe_forward_path.
 *   logits       device float [T][E]
 *   topk_ids     device int32 [T][k] (output)
 *   topk_weights device float [T][k] (output)
 * Limits: E <= 1024, k <= 32.  Errors: as pw_moe_forward_path. */
int pw_moe_forward_logits(const pw_moe_shape* shape, const void* hidden, const float* logits,
                          int32_t* topk_ids, float* topk_weights, const pw_page_table* table,
                          float* out, void* workspace, size_t workspace_bytes, int32_t path,
                          cudaStream_t stream);

/* Token count from which PW_PATH_AUTO takes the prefill path for a shape
 * (T*k pairs >= this value). */
int32_t pw_prefill_min_pairs(const pw_moe_shape* shape);

/* ---- measurement hook ---------------------------------------------------------
 * No counterpart on the PagedWeight pages: a benchmark needs the duration of
 * the call's dominant kernel, which the caller cannot bracket from outside.
 * While set, every forward call records `before` on its stream right before
 * it launches its dominant kernel and `after` right after it: the decode
 * path's gate_up kernel, the prefill path's gate_up GEMM.  During stream
 * capture the records become external event-record nodes of the graph.
 * The events must have timing enabled; pass NULL, NULL to stop.  Process-wide
 * and not thread-safe.  Errors: PW_ERR_INVALID_ARG (exactly one is NULL). */
int pw_set_timing_events(cudaEvent_t before, cudaEvent_t after);

/* ---- checks of the kernels' own code -----------------------------------------
 * No counterpart on the PagedWeight pages: these run pieces of the forward
 * kernels' device code on whole blocks and write the results back in plain
 * order, so that tests can compare them bit for bit with the format's
 * definition (PagedWeight, "Core components" 1: a b-bit view reads the top b
 * planes, idx = code >> (8 - b); the weight is the row's LUT entry).
 *
 * Index forms the kernels rebuild indices in: */
#define PW_INDEX_NIBBLES 0  /* decode kernels, q <= 4 (pair-table lookups)          */
#define PW_INDEX_BYTES   1  /* decode kernels, q = 5, 6, 8 (any q)                  */
#define PW_INDEX_HALVES  2  /* tensor-core dequant warps (16-column halves)          */

/* idx[n][k] = the index the kernels' extraction code produces for column k of
 * row n of a block read at bitwidth q in the given form.
 *   planes device uint32 [>= q][K/32][N];  idx device uint8 [N][K] (output)
 * Errors: PW_ERR_INVALID_ARG, PW_ERR_SHAPE (K % 32), PW_ERR_UNSUPPORTED_Q (q
 * off the ladder; q > 4 with PW_INDEX_NIBBLES). */
int pw_debug_index(const uint32_t* planes, int32_t N, int32_t K, int32_t q, int32_t form,
                   uint8_t* idx, cudaStream_t stream);

/* w[n][k] = the weight the kernels' table build and lookup give for column k
 * of row n at bitwidth q, widened to float: path PW_PATH_DECODE builds the
 * decode kernels' tables (fp32 tables for q = 5, 6, 8; fp16 pair tables for
 * q = 3, 4) pass by pass as the kernels do; PW_PATH_PREFILL the dequant
 * warps' fp16 LUT layout.
 *   planes device uint32 [>= q][K/32][N];  lut device fp16 [N][2^q] (16-byte
 *   aligned);  w device float [N][K] (output);  table (may be NULL): its status
 *   word receives PW_ERR_RANGE for a LUT value a pair table cannot hold
 * Errors: PW_ERR_INVALID_ARG, PW_ERR_SHAPE (K % 32, N % 32), PW_ERR_UNSUPPORTED_Q. */
int pw_debug_dequant(const uint32_t* planes, const uint16_t* lut, int32_t N, int32_t K, int32_t q,
                     int32_t path, float* w, pw_page_table* table, cudaStream_t stream);

/* Byte range [*offset, *offset + *bytes) of a forward call's workspace that
 * holds, after the call (path PW_PATH_DECODE / PW_PATH_PREFILL):
 *   section 0: offsets int32 [E+1] of the grouping by expert;
 *   section 1: perm int32 [T*k], the grouped pair ids;
 *   section 2: decode: the hidden states in the kernels' fp32 form, float
 *              [T][H], column c of each group of 32 at 4 (c % 8) + c / 8;
 *              prefill: the gathered rows, fp16 [T*k][H] (grouped order),
 *              each scaled by 2^-e of its row;
 *   section 3: decode: the fp16 records, 80 bytes per (token, group of 32
 *              columns): 32 fp16 x * 2^-e at 8 (c % 4) + 2 (c / 8) + (c / 4) % 2,
 *              the floats 2^e of columns 0-15 and 16-31 at bytes 64 and 68;
 *              prefill: the row scales 2^e, float [T*k].
 * Errors: PW_ERR_INVALID_ARG (unknown path or section, NULL), shape errors. */
int pw_debug_workspace_section(const pw_moe_shape* shape, int32_t path, int32_t section,
                               size_t* offset, size_t* bytes);

/* ---- failure-detection check -------------------------------------------------
 * No counterpart on the PagedWeight pages.  Every device-side wait of the
 * forward kernels is bounded so that a wait that can never end (a producer
 * that stopped, a barrier nobody arrives at) costs a status code, not a hung
 * GPU.  This entry point proves that on the device without starving a real
 * forward call: it runs one of those waits, the same device code with a
 * caller-chosen limit, against something that is never released:
 *   which 0: the decode down kernel's wait for an expert's gate_up tiles,
 *            on a counter nothing increments (each poll sleeps ~128 ns);
 *   which 1: the tensor-core kernels' mbarrier wait, on a barrier whose
 *            phase never completes.
 * After `polls` polls the wait gives up, latches PW_ERR_TIMEOUT in the table's
 * status word (read with pw_page_table_status) and the kernel returns; the
 * context stays usable.  Errors: PW_ERR_INVALID_ARG (NULL table, which not 0
 * or 1, polls outside 1..2^20), PW_ERR_UNSUPPORTED_DEVICE, PW_ERR_CUDA. */
int pw_debug_bounded_wait(pw_page_table* table, int32_t which, int32_t polls,
                          cudaStream_t stream);

/* Pipeline trace of the tensor-core gate_up GEMM, a measurement hook with no
 * counterpart on the pages.  A library built with tracing (build.py --trace,
 * which writes libpw_trace.so) records %globaltimer stamps (nanoseconds) in the
 * gate_up GEMM launches of both the prefill path and the decode path's heavy
 * experts, for CTAs 0, 10, 20, ... 150 (trace slot = block index / 10); the
 * record is cleared before each such launch, so it holds the last one.  This
 * call copies it (synchronously) into host memory laid out as, in this order,
 *   uint64 step[16][256][4]: for the CTA's first 256 k-steps (its ring
 *          position): [0] the MMA issuer found the stage full, [1] it had
 *          issued the stage's MMAs and commit, [2] a dequant set had written
 *          and announced the stage's A rows, [3] the token producer found the
 *          stage empty (0: not reached);
 *   uint64 dq[16][256][8][4]: per k-step and warp of the dequant set that owns
 *          it: [0] the warp's wait for the stage's release done, [1] its
 *          announcement of the stage's A rows done, [2] its wait for the
 *          plane words done, [3] its index transpose done;
 *   uint64 tile[16][32][6]: for the CTA's first 32 tiles: [0] MMA start (the
 *          accumulator free), [1] last commit, [2] epilogue start, [3]
 *          epilogue end, [4] LUT load start, [5] LUT load end;
 *   uint64 smid[16]: the SM the CTA ran on, plus one (0: no such CTA).
 *   host    host buffer of at least *needed bytes
 *   needed  (may be NULL) receives the record's size
 * Errors: PW_ERR_INVALID_ARG (NULL or short buffer), PW_ERR_NOT_BUILT (built
 * without tracing), PW_ERR_UNSUPPORTED_DEVICE, PW_ERR_CUDA. */
int pw_debug_gemm_trace(void* host, size_t bytes, size_t* needed);

/* Per-tile phase trace of the decode gate_up kernel, a measurement hook with
 * no counterpart on the pages.  A library built with tracing (build.py
 * --trace) records, in each decode gate_up launch, for CTAs 0, 19, 38, ...
 * 285 (trace slot = block index / 19) and their first 32 tiles, where thread
 * 0 of the CTA spent its time; the record is cleared before each launch, so
 * it holds the last one.  This call copies it (synchronously) into host
 * memory laid out as, in this order,
 *   uint64 tile[16][32][10]: [0] tile start and [1] tile end (%globaltimer
 *          ns; 0: not reached); SM cycles (clock64) spent on [2] the slot
 *          descriptor (with the release of the previous tile's h rows), [3]
 *          the passes' set-up (LUT fetch, first copies of the ring, table
 *          build), [4] the token groups' column loops up to the barrier after
 *          the partial sums, [5] their reduction, SiLU and h stores; [6] the
 *          tile's q + 256 * its number of pairs; the parts of [3]: [7]
 *          issuing the LUT loads and first ring copies, [8] waiting for
 *          thread 0's LUT words and building its share of the tables, [9]
 *          the barrier after the build;
 *   uint64 cta[16][2]: the SM the CTA ran on plus one (0: no such CTA), and
 *          its exit time (ns).
 *   host    host buffer of at least *needed bytes
 *   needed  (may be NULL) receives the record's size
 * Errors: PW_ERR_INVALID_ARG (NULL or short buffer), PW_ERR_NOT_BUILT (built
 * without tracing), PW_ERR_UNSUPPORTED_DEVICE, PW_ERR_CUDA. */
int pw_debug_decode_trace(void* host, size_t bytes, size_t* needed);

/* ---- the fused layer without a workspace ------------------------------------
 * The PagedWeight pages have no counterpart to this entry point; it is a
 * service for callers that cannot allocate device memory: a plugin whose
 * enqueue hook only receives its input and output buffers, a runtime that
 * fixes its memory budget at start-up and allows no allocation afterwards, or
 * code where a cudaMalloc would synchronise the device or break a capture.
 *
 * Same function and arguments as pw_moe_forward on the decode path, minus the
 * workspace: the scratch lives in one static device array of 8 MiB inside
 * libpw (every GPU that loads the library keeps those 8 MiB until the process
 * exits).  The caller still passes inputs and outputs.
 *   - Shapes whose decode scratch, about 6.5*T*H + T*k*(6.5*I + 4*H + 4)
 *     + 116*E + H/8 bytes, plus 4*T*k*H when I >= 8192 (each section
 *     rounded up to 256 bytes), exceeds
 *     8 MiB are rejected with
 *     PW_ERR_WORKSPACE (use pw_moe_forward with a workspace instead), as
 *     are shapes beyond the decode path's limits (PW_ERR_SHAPE).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - The call allocates nothing: no cudaMalloc, no cudaFree.  Each call
 *     zeroes the counters it needs and writes every other scratch byte before
 *     reading it, so nothing is carried over from an earlier call.
 *   - All calls on a device share the one array: calls that can overlap on
 *     the GPU (different streams without ordering) race on it and produce
 *     wrong results.  Order them on one stream.
 * Errors: as pw_moe_forward, plus PW_ERR_WORKSPACE for shapes over the limit. */
int pw_moe_forward_noalloc(const pw_moe_shape* shape, const void* hidden,
                           const int32_t* topk_ids, const float* topk_weights,
                           const pw_page_table* table, float* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PW_H_ */
