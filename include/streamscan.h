/*
 * streamscan.h -- C ABI of libstreamscan.so: device-wide prefix sums and
 * order-preserving stream compaction on one NVIDIA GB300 (sm_103a).
 *
 * Definitions ("Prefix sum and other parallel patterns", Definitions):
 *   inclusive  out[i] = in[0] + ... + in[i]
 *   exclusive  out[i] = in[0] + ... + in[i-1],  out[0] = 0
 * e.g. in = [3,1,7,0,4,1,6,3] gives inclusive [3,4,11,11,15,16,22,25] and
 * exclusive [0,3,4,11,11,15,16,22].
 *
 * Conventions shared by every call:
 *   - Pointers named in/out/keys/flags/d_count/d_carry_* are DEVICE
 *     pointers owned by the caller (e.g. from torch, cudaMalloc).  Pointers
 *     named h_* are HOST pointers.  The library never frees caller memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device
 *     calls only enqueue work and return; results are ready when the stream
 *     reaches them.  Calls on one stream run in order; calls on different
 *     streams are independent (each (device, stream) pair has its own
 *     workspace).
 *   - int32 and uint32 sums wrap modulo 2^32 (two's complement for int32).
 *     fp32 sums use IEEE round-to-nearest adds in an order the caller does
 *     not control; the last bits of an fp32 result may differ from run to
 *     run, because a tile adds its predecessors' published sums in whatever
 *     grouping the look-back found.
 *   - 16-byte aligned in/out take the vectorised path; any 4-byte aligned
 *     pointers are accepted and take a slower element-wise path.
 *   - Argument errors are found before anything is enqueued and return
 *     SS_ERR_INVALID_ARG (ss_last_error_detail() says why).  Launch
 *     failures return SS_ERR_CUDA.  Errors found on the device (a look-back
 *     wait that ran out) are recorded in the stream's status word and
 *     returned by the next ss_stream_status() call on that stream; the
 *     outputs of the failing call are then undefined.
 *   - n == 0 is a valid no-op (the compactions still write *d_count = 0).
 *   - The library owns a small per-(device, stream) workspace (tile
 *     descriptors, a tile counter, the status word), about 8 bytes per 4096
 *     elements, grown on demand with stream-ordered allocation and freed
 *     by ss_shutdown().  Size it before capturing a stream into a CUDA
 *     graph by making one call of the largest n on that stream first; a
 *     captured graph may then be replayed any number of times up to 2^29
 *     (the device-side launch epoch separates the replays).
 */
#ifndef STREAMSCAN_H
#define STREAMSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that the header needs no CUDA
 * include. */
typedef struct CUstream_st *ss_stream_t;

typedef enum ss_status {
    SS_OK = 0,
    SS_ERR_INVALID_ARG = 1,      /* bad pointer, size or overlap */
    SS_ERR_CUDA = 2,             /* a CUDA runtime call or launch failed */
    SS_ERR_LOOKBACK_TIMEOUT = 3, /* a tile's look-back wait ran out */
    SS_ERR_NO_MEMORY = 4,        /* workspace allocation failed */
    SS_ERR_UNSUPPORTED = 5       /* no usable device, or bad enum value */
} ss_status;

typedef enum ss_dtype { SS_I32 = 0, SS_U32 = 1, SS_F32 = 2 } ss_dtype;

/* Algorithms for ss_scan().  SS_ALGO_LOOKBACK is the product path; the
 * others are the measured ablations. */
typedef enum ss_algo {
    SS_ALGO_LOOKBACK = 0,            /* single pass, decoupled look-back, 2n traffic */
    SS_ALGO_REDUCE_THEN_SCAN = 1,    /* three kernels, 3n traffic */
    SS_ALGO_RTS_BLELLOCH = 2,        /* same, third kernel a Blelloch tree, unpadded */
    SS_ALGO_RTS_BLELLOCH_PAD32 = 3,  /* same, tree padded i + i/32 */
    SS_ALGO_RTS_BLELLOCH_PAD2 = 4    /* same, tree padded i + i/32 + i/1024 */
} ss_algo;

/*
 * Device-wide scans, single pass with decoupled look-back ("Prefix sum and
 * other parallel patterns", A device-level scan: scan then propagate --
 * each block looks back at the states earlier blocks published, "local sum
 * only" or "inclusive prefix available").
 *   in   device, n elements, read once.
 *   out  device, n elements, written once.  out == in is allowed (in-place);
 *        any other overlap is SS_ERR_INVALID_ARG.
 *   n    element count, 0 <= n < 2^31 * 4096.
 */
ss_status scan_inclusive_i32(const int32_t *in, int32_t *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_i32(const int32_t *in, int32_t *out, size_t n, ss_stream_t stream);
ss_status scan_inclusive_u32(const uint32_t *in, uint32_t *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_u32(const uint32_t *in, uint32_t *out, size_t n, ss_stream_t stream);
ss_status scan_inclusive_f32(const float *in, float *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_f32(const float *in, float *out, size_t n, ss_stream_t stream);

/*
 * Scans with 64-bit sums ("Parallel Prefix Sum (Scan) for NVIDIA T4
 * (sm_75)", Key Features: 64-bit indexing for large arrays; the sum of many
 * 32-bit counts needs 64 bits).  Same definitions and method as the 32-bit
 * scans, with 16-byte tile descriptors.
 *   u32_u64  uint32 in, uint64 out: the exact sums (no wrap below 2^64).
 *   i32_i64  (ss_scan_wide only) int32 in, int64 out: the exact sums.
 *   i64      int64 in and out, wrapping modulo 2^64 (uint64 data gives the
 *            same bits).
 *   f64      fp64 in and out, IEEE round-to-nearest adds in an order the
 *            caller does not control (as for fp32).
 *   in   device, n elements, aligned to the element size (16-byte aligned
 *        in and out take the bulk-copy path; for f64, the tensor-copy path).
 *   out  device, n 8-byte elements.  out == in is allowed for i64 and f64;
 *        any other overlap is SS_ERR_INVALID_ARG.
 *   n    0 <= n < 2^31 * 8192.
 */
typedef enum ss_wide_type {
    SS_WIDE_U32_U64 = 0,
    SS_WIDE_I32_I64 = 1,
    SS_WIDE_I64 = 2,
    SS_WIDE_F64 = 3
} ss_wide_type;
ss_status scan_inclusive_u32_u64(const uint32_t *in, uint64_t *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_u32_u64(const uint32_t *in, uint64_t *out, size_t n, ss_stream_t stream);
ss_status scan_inclusive_i64(const int64_t *in, int64_t *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_i64(const int64_t *in, int64_t *out, size_t n, ss_stream_t stream);
ss_status scan_inclusive_f64(const double *in, double *out, size_t n, ss_stream_t stream);
ss_status scan_exclusive_f64(const double *in, double *out, size_t n, ss_stream_t stream);
ss_status ss_scan_wide(ss_wide_type type, int inclusive, const void *in, void *out, size_t n,
                       ss_stream_t stream);

/*
 * Order-preserving stream compaction in one pass: out receives, in index
 * order, every keys[i] whose flags[i] != 0, and *d_count the number kept
 * ("Prefix sum and other parallel patterns", Stream compaction and
 * Exercise 1: out[pos[i]] = in[i] with pos the exclusive scan of the 0/1
 * keep flags, count = pos[n-1] + flags[n-1]; fused so that the flags' scan
 * and the positions never reach device memory).
 *   keys     device, n uint32.
 *   flags    device, n uint8; any nonzero byte keeps the element.
 *   out      device, room for n uint32 (only the first *d_count written);
 *            must not overlap keys or flags.
 *   d_count  device, one uint64, written by the call.
 *   n        0 <= n < 2^32.
 */
ss_status compact_u32(const uint32_t *keys, const uint8_t *flags, uint32_t *out,
                      uint64_t *d_count, size_t n, ss_stream_t stream);

/*
 * Order-preserving compaction with a built-in predicate instead of a flag
 * array: out receives, in index order, every in[i] with in[i] > 0, and
 * *d_count the number kept ("Prefix sum and other parallel patterns",
 * Stream compaction, compact.cu's predicate v > 0, and Exercise 1's flags
 * in[i] > 0 fused into the scan's passes).  The predicate is evaluated in
 * the element type: for fp32, NaN, +0.0 and -0.0 are dropped and +inf is
 * kept; for int32 it is signed; for uint32 it means nonzero.  Kept elements
 * are copied bit for bit.
 *   in       device, n elements of `dtype`, read once.
 *   out      device, room for n elements (only the first *d_count written);
 *            must not overlap in.
 *   d_count  device, one uint64, written by the call.
 *   n        0 <= n < 2^32.
 * Errors as compact_u32.
 */
ss_status compact_positive_f32(const float *in, float *out, uint64_t *d_count, size_t n, ss_stream_t stream);
ss_status ss_compact_positive(ss_dtype dtype, const void *in, void *out, uint64_t *d_count, size_t n,
                              ss_stream_t stream);

/*
 * Unordered compaction (the measured ablation): the same kept elements and
 * count as compact_u32 / ss_compact_positive, but in no fixed order.  Each
 * warp claims room for its kept elements with one atomic add on *d_count
 * and writes them at the claimed offset plus their rank inside the warp
 * ("Prefix sum and other parallel patterns", Stream compaction: the
 * warp-aggregated atomic, ballot and popc).  Within each 512-element batch
 * of a warp the order is kept; the order of the batches depends on the
 * timing of the atomics.  Needs no workspace and no look-back.  *d_count is
 * zeroed on the stream first, then counted up by the kernel.  Arguments and
 * errors as the ordered calls.
 */
ss_status ss_compact_u32_unordered(const uint32_t *keys, const uint8_t *flags, uint32_t *out,
                                   uint64_t *d_count, size_t n, ss_stream_t stream);
ss_status ss_compact_positive_unordered(ss_dtype dtype, const void *in, void *out, uint64_t *d_count,
                                        size_t n, ss_stream_t stream);

/*
 * Batched scans: every row of a row-major rows x cols matrix scanned on its
 * own, the sum starting from zero at each row (for example the cumulative
 * sum over each row's sorted probabilities in top-p sampling, "Prefix sum
 * and other parallel patterns", In LLMs: MoE token dispatch, last
 * paragraph).  Same element types, wraparound and fp32 rules as the flat
 * scans.
 *   in    device, rows * cols elements, row r at in + r * cols.
 *   out   device, same shape; out == in is allowed, any other overlap is
 *         SS_ERR_INVALID_ARG.
 *   rows, cols  either may be 0 (a no-op); rows * cols < 2^31 * 4096, and
 *         for rows longer than 2048 elements rows * ceil(cols / 4096) < 2^31.
 * Rows longer than 2048 elements use row-aligned tiles with the decoupled
 * look-back (the per-stream workspace); shorter rows take one warp each;
 * rows of 2^21 elements or more run as one flat scan each.
 */
ss_status ss_scan_rows(ss_dtype dtype, int inclusive, const void *in, void *out, size_t rows, size_t cols,
                       ss_stream_t stream);

/*
 * Segmented scans: every segment [offsets[s], offsets[s+1]) of a flat array
 * scanned on its own, from zero; the general form of ss_scan_rows, for rows
 * of different lengths.  Same element types, wraparound and fp32 rules as the
 * flat scans.
 *   in, out       device, n elements each; out == in is allowed, any other
 *                 overlap is SS_ERR_INVALID_ARG.
 *   d_offsets     device, num_segments + 1 uint64: offsets[0] = 0,
 *                 non-decreasing, offsets[num_segments] = n (empty segments
 *                 are fine).  Only the starts offsets[0 .. num_segments-1]
 *                 are read, and the scan restarts at each start below n (so
 *                 with offsets as described the result is the definition
 *                 above).
 *   num_segments  0 means one segment, the whole array.
 * Two launches on the stream: a pass that marks the segment starts in a
 * workspace bitmask (n / 8 bytes), then the single-pass scan with a
 * segmented add, in which a tile holding a segment start publishes its
 * inclusive prefix at once.
 */
ss_status ss_scan_segments(ss_dtype dtype, int inclusive, const void *in, void *out, size_t n,
                           const uint64_t *d_offsets, size_t num_segments, ss_stream_t stream);

/*
 * MoE token counts and expert offsets aligned to GEMM tiles ("Prefix sum and
 * other parallel patterns", In LLMs: MoE token dispatch, steps 1-2, and
 * Exercise 2: a histogram of the router's expert ids, then an exclusive
 * prefix sum for each expert's start, each expert's segment rounded up to a
 * multiple of the tile size):
 *   counts[e]    = number of i < m with topk_ids[i] == e
 *   offsets[0]   = 0,  offsets[e+1] = offsets[e] + align * ceil(counts[e] / align)
 * An id outside [0, num_experts) is counted nowhere.
 *   topk_ids     device, m int32 (a row-major num_tokens x top_k array, flat).
 *   m            number of ids, 0 <= m < 2^31.
 *   num_experts  E, 1 <= E <= 16384.
 *   align        tile size, 1 <= align <= 2^20 (1 gives the plain exclusive
 *                scan of the counts); m + E * (align - 1) must fit 32 bits.
 *   d_counts     device, E uint32, written.
 *   d_offsets    device, E + 1 uint32, written (offsets[E] = padded total).
 * One kernel launch; no allocation after the stream's first call with this
 * E and grid size.  Arrays must not overlap.
 */
ss_status ss_moe_counts_offsets(const int32_t *topk_ids, size_t m, int32_t num_experts, uint32_t align,
                                uint32_t *d_counts, uint32_t *d_offsets, ss_stream_t stream);

/*
 * Generic scan entry: dtype, inclusive (0/1) and algorithm chosen at run
 * time.  Same argument rules as the named scans.  The reduce-then-scan
 * algorithms ("Prefix sum and other parallel patterns", three passes with
 * scan_block_sums' carry loop; "The CUDA scan algorithm: the tree and the
 * three kernels", Two sweeps over one tree, bank padding of "The stride
 * doubles, and so does the conflict") also take out == in.
 */
ss_status ss_scan(ss_dtype dtype, int inclusive, ss_algo algo, const void *in, void *out,
                  size_t n, ss_stream_t stream);

/*
 * Sum of all n elements of `in`, written to *d_total (device, one element of
 * dtype's type, 4-byte aligned) -- the first step of a scan split over
 * several devices ("Prefix sum and other parallel patterns", A device-level
 * scan: scan then propagate -- the part totals are scanned and each part is
 * offset by the sum of the parts before it).  int32 and uint32 wrap modulo
 * 2^32; fp32 adds in an order that is fixed for a fixed n and device (so the
 * same input gives the same bits on every run).  n == 0 writes 0.  in is
 * 4-byte aligned (16-byte aligned takes the vector path); *d_total must not
 * overlap in.  One launch; uses the stream's workspace.
 */
ss_status ss_reduce_sum(ss_dtype dtype, const void *in, void *d_total, size_t n, ss_stream_t stream);

/*
 * Single-pass scan seeded with a carry: the prefix before in[0] is
 * *d_carry_in (device, one element of the scan's type; NULL means 0), and
 * the inclusive total including the seed is written to *d_carry_out (device,
 * NULL to skip).  Scanning an array in consecutive chunks with the carry
 * passed along gives the scan of the whole array; this is the offset step of
 * a scan split over several calls or several devices (scan each part, scan
 * the parts' totals, seed each part with its offset).  d_carry_out may
 * equal d_carry_in.
 */
ss_status ss_scan_seeded(ss_dtype dtype, int inclusive, const void *in, void *out, size_t n,
                         const void *d_carry_in, void *d_carry_out, ss_stream_t stream);

/*
 * Host-memory scan: h_in and h_out are HOST pointers.  Returns when h_out
 * holds the result (device errors are reported directly).  h_out == h_in is
 * allowed.  Two paths:
 *   - both buffers pinned and mapped into the device address space (for
 *     example from cudaHostAlloc): the scan kernel reads h_in and writes
 *     h_out directly, over NVLink-C2C on a Grace host, with no staging
 *     copies.  It uses the one-CTA-per-tile kernel, whose accesses are plain
 *     16-byte loads and stores;
 *   - otherwise (pageable memory, or ss_set_host_mode(1)): the input is
 *     copied to the device in chunks, each chunk is scanned seeded with the
 *     running carry, and the results are copied back, the copies of one chunk
 *     overlapping the scan of another.
 */
ss_status ss_scan_host(ss_dtype dtype, int inclusive, const void *h_in, void *h_out, size_t n,
                       ss_stream_t stream);

/* Path of ss_scan_host: 0 (default) = direct access when both buffers are
 * mapped pinned memory, else staged; 1 = always staged.  Process-wide. */
ss_status ss_set_host_mode(int mode);

/*
 * Bandwidth probe: copies n uint32 from in to out with the scan's loader and
 * storer and no arithmetic ("The CUDA scan algorithm: the tree and the three
 * kernels", Results: "copy, no scan" as the speed-of-light row).
 */
ss_status ss_copy_u32(const uint32_t *in, uint32_t *out, size_t n, ss_stream_t stream);

/*
 * Diagnostic: the exclusive uint32 (= int32 bits) single-pass scan under
 * tile configuration `config`, recording a timing trace of every tile's
 * look-back ("Prefix sum and other parallel patterns", A device-level scan:
 * how long a tile waits on what earlier tiles published).  d_trace (device,
 * 8-byte aligned) receives 8 uint64 per tile of that configuration
 * (ss_scan_tile_elems() after ss_set_scan_config(config)):
 *   [0] %globaltimer (ns) when the CTA began the tile  [1] aggregate known
 *   [2] aggregate published   [3] look-back resolved   [4] outputs issued
 *   [5] descriptor windows read   [6] polls that found an unpublished tile
 *   [7] SM id (low 32 bits) | CTA index << 32
 * Every row has a traced build (rows 10-12, with the two-level look-back,
 * record [5] = 1).  A persistent row needs 16-byte aligned in/out and n
 * above one tile.  The scan result is the same as scan_exclusive_u32's.
 */
ss_status ss_scan_trace(int config, const uint32_t *in, uint32_t *out, size_t n, uint64_t *d_trace,
                        ss_stream_t stream);

/*
 * Waits for `stream`, then returns and clears the device-side status of
 * that stream's workspace: SS_OK, SS_ERR_LOOKBACK_TIMEOUT, or SS_ERR_CUDA if
 * the stream itself failed.  *failing_tile (may be NULL) receives the first
 * tile that gave up, or -1.
 */
ss_status ss_stream_status(ss_stream_t stream, int64_t *failing_tile);

/* Static description of a status code. */
const char *ss_status_string(ss_status status);

/* Detail of the last error returned on the calling thread ("" if none). */
const char *ss_last_error_detail(void);

/* Elements per tile of the single-pass scan under the current tile
 * configuration (under the automatic choice, of the row used for large n),
 * and the number of configurations that can be selected. */
size_t ss_scan_tile_elems(void);
int ss_scan_config_count(void);

/* Selects the single-pass scan's tile configuration for later calls in this
 * process (ss_scan_config_count() rows: one CTA per tile, or a persistent
 * grid streaming tiles through a shared-memory ring).  -1 (the initial
 * setting) chooses per call by size: row 7 (16384-element tiles) from 2e6
 * to 5e7 elements, row 8 (18432-element tiles, each claimed from the tile
 * counter as its copy starts, so that faster SMs take more tiles) below and
 * above.
 * Results do not depend on it, except for the rounding of fp32 sums.
 * SS_ERR_INVALID_ARG below -1 or from ss_scan_config_count() on. */
ss_status ss_set_scan_config(int config);

/* Selects the persistent compaction kernel used for 16-byte aligned inputs
 * above 16384 elements (flag form), for later calls in this process:
 *   0  streams keys and flags through shared memory with bulk copies;
 *   1  bulk-copies only the flags and loads a 16-byte key vector only where
 *      one of its four flags is set, which reads far fewer key bytes when
 *      few elements are kept; one look-back per 16384 elements;
 *   2  (the default) as 1, with one look-back per tile of four chunks: two
 *      256-thread CTAs per SM and 32768-element tiles, which pays a tile's
 *      fixed costs once per 32768 elements (inputs of 32768 elements or
 *      fewer take 1).  A tile keeping fewer than 1728 keys is written in a
 *      sparse form: each thread loads only its kept keys, one by one, before
 *      the tile's look-back; other tiles gather each warp's kept keys in
 *      shared memory and write 16-byte vectors;
 *   3  as 2 with every tile in the dense form, 4 with every tile in the
 *      sparse form;
 *   5, 6, 7  as 2, 3, 4 with one 512-thread CTA per SM and 65536-element
 *      tiles (sparse below 3456 keys).
 * Results are identical. */
ss_status ss_set_compact_config(int config);

/* Selects the form of later ss_scan_segments calls in this process:
 *   0  (the default) blocked, by mean segment length n / num_segments: 64
 *      threads a CTA below 2048, 128 from there and for num_segments = 0;
 *   1  row-striped: lane l of a warp holds 16-byte vectors l, l + 32, ... of
 *      the warp's span, one 512-thread CTA per SM, 16384-element tiles;
 *   2, 3, 4, 5  blocked: each thread owns 32 consecutive elements (one
 *      tile row), with 256, 128, 512 or 64 threads a CTA, 512 / threads CTAs
 *      per SM and tiles of 32 x threads elements.
 * Integer results are identical; fp32 sums are added in another order and
 * agree within the bound of the flat scans.  SS_ERR_INVALID_ARG for any
 * other value. */
ss_status ss_set_segments_config(int config);

/* Frees every workspace the library allocated (all devices and streams).
 * No call may be in flight. */
void ss_shutdown(void);

/*
 * Test hook for the failure path of the look-back wait.  With tile >= 0,
 * later single-pass calls in this process skip publishing that tile's
 * descriptor, so its successors' waits run out after timeout_ns (their
 * status then reads SS_ERR_LOOKBACK_TIMEOUT).  tile = -1 restores normal
 * operation and timeout_ns = 0 restores the default limit (2 s).  No wait is
 * ever unbounded: every wait also stops after a fixed number of polls.
 */
ss_status ss_debug_set_lookback_fault(int64_t tile, uint64_t timeout_ns);

/*
 * Single-pass scan that allocates nothing.  The pages have no counterpart:
 * it exists for callers that cannot call cudaMalloc -- an application that
 * serves all device memory from its own pool and forbids other allocations
 * to keep its accounting exact, or a latency-critical loop that may never
 * pay for an allocation.  The regular entry points allocate a per-stream
 * workspace on first use; this one keeps its scratch (tile counter, status
 * words, tile descriptors) in a fixed device array of 2 MiB + 256 bytes that
 * every GPU loading the library holds until the process exits.
 *   dtype, inclusive, in, out, stream: as for ss_scan (SS_ALGO_LOOKBACK);
 *        out == in is allowed.  The caller passes inputs and outputs.
 *        `stream` must belong to the current device (the array used is the
 *        current device's); a stream of another device returns
 *        SS_ERR_INVALID_ARG.
 *   n    0 <= n <= 2^30; larger n returns SS_ERR_INVALID_ARG.
 * The first call on a device sets up that device: it looks up the array's
 * device address and zeroes it, which synchronises the device; make that
 * first call before any stream capture.  Every call on a device shares the
 * array and keeps the previous call's contents; no per-call clearing is
 * needed (descriptors carry a launch epoch and the tile counter returns to
 * zero at the end of each launch).  Calls that overlap on the GPU race on
 * the shared array: serialise them (one stream, or events).  The returned
 * status is the only error report: device-side look-back timeouts are not
 * read back by this entry point, nor reported by ss_stream_status().
 */
ss_status ss_scan_noalloc(ss_dtype dtype, int inclusive, const void *in, void *out, size_t n,
                          ss_stream_t stream);

/*
 * Explicit-workspace form, in CUB's two-call shape ("Prefix sum and other
 * parallel patterns", Stream compaction: the library call that first asks
 * for its temporary storage size, then runs with the caller's buffer).
 *
 * ss_scan_temp_bytes: *bytes receives the device scratch, in bytes, that a
 *   scan of n elements needs: a 256-byte header (the tile counter and the
 *   status words) and 8 bytes per 4096 elements and per 32 tiles of them
 *   (the tile descriptors); 0 for n = 0.  Host only; enqueues nothing.
 *
 * ss_scan_ws: the scan of scan_{inclusive,exclusive}_* (dtype SS_I32,
 *   SS_U32 or SS_F32; the same kernels and the same automatic choice by n)
 *   with `temp` as its scratch instead of the library's per-stream
 *   workspace, so the call allocates nothing.
 *   temp        device memory of the stream's device, 256-byte aligned, at
 *               least ss_scan_temp_bytes(n) bytes (temp_bytes), owned by the
 *               caller and not overlapping in or out.  Its contents on entry
 *               do not matter: the call clears the part it uses with one
 *               memset on `stream` before its launch.
 *   in, out, n, stream: as for the scans above; out == in is allowed.
 *   Calls sharing one temp must not overlap on the GPU.  Device-side
 *   timeouts are recorded in temp's header: ss_temp_status reads them.
 *
 * ss_temp_status: waits for `stream`, then returns and clears the device
 *   status held in `temp` (the values of ss_stream_status); *failing_tile
 *   (may be NULL) receives the first tile that gave up, or -1.
 */
ss_status ss_scan_temp_bytes(size_t n, size_t *bytes);
ss_status ss_scan_ws(ss_dtype dtype, int inclusive, const void *in, void *out, size_t n, void *temp,
                     size_t temp_bytes, ss_stream_t stream);
ss_status ss_temp_status(void *temp, ss_stream_t stream, int64_t *failing_tile);

/*
 * Test hooks for ss_scan_noalloc's periodic descriptor clear: the clear runs
 * on the current device's call that makes the count of calls a multiple of
 * ss_debug_noalloc_clear_period() (2^29), before its launch.
 * ss_debug_set_noalloc_calls sets the count of calls made so far on the
 * current device, so that a test reaches a clear in a few calls.
 */
ss_status ss_debug_set_noalloc_calls(uint64_t calls);
uint64_t ss_debug_noalloc_clear_period(void);

#ifdef __cplusplus
}
#endif

#endif /* STREAMSCAN_H */
