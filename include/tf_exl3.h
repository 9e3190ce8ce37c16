/*
 * tf_exl3.h -- C ABI of the GB300 (sm_103a) trellis-quantized projection for
 * decode rows: the input rotation (rot_in) and the trellis linear.
 *
 * Source of the method: "hip exl3: the input rotation and trellis linear for
 * decode rows, under the kernel contract" (TensorFold pull request #3314),
 * section "What this changes". Callers issue rot_in and then the linear for
 * each projection; the linear has no bias and no split of the inner sums
 * exposed to the caller, and takes 1 to 16 rows a pass and any number of
 * passes.
 *
 * Conventions shared by every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller (for example
 *     allocated by PyTorch). Row-major layouts; sizes in elements unless said.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous on that stream; nothing synchronises.
 *   - The current CUDA device is used; pointers must belong to it.
 *   - Arguments are checked before any launch. A refused call returns a
 *     non-zero tf_status, launches nothing and writes nothing. No call traps.
 *   - tf_trellis_linear keeps a per-device workspace (about 30 MB on a
 *     152-SM GPU) for partial sums of output blocks; it is allocated on the
 *     first call on each device (call once before capturing a CUDA graph) and
 *     reused, never per call.
 *   - Thread safety: calls may come from several host threads.
 */
#ifndef TF_EXL3_H
#define TF_EXL3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TF_OK = 0,
  TF_ERR_NULL = 1,     /* a required pointer is NULL                          */
  TF_ERR_SHAPE = 2,    /* rows < 0, or in/out features not positive multiples of 128 */
  TF_ERR_BITS = 3,     /* bits not in {2, 3, 4, 5, 6, 8}                       */
  TF_ERR_DTYPE = 4,    /* unsupported dtype code                               */
  TF_ERR_ALIGN = 5,    /* a pointer is not 16-byte aligned                     */
  TF_ERR_CUDA = 6,     /* a CUDA runtime call or launch failed (tf_last_error) */
  TF_ERR_TIMEOUT = 7,  /* a kernel's bounded wait expired (tf_device_error)    */
  TF_ERR_POINTER = 8,  /* a pointer is not device memory of the current device */
  TF_ERR_SCRATCH = 9   /* the problem needs more scratch than the given workspace or the no-allocation array holds */
} tf_status;

typedef enum { TF_F16 = 0, TF_F32 = 1, TF_BF16 = 2 } tf_dtype;

/* Version of this ABI (incremented on any incompatible change). The pages
 * have no counterpart: it is this library's own. */
int tf_abi_version(void);

/*
 * tf_rot_in -- rotate activation rows by 128 ("What this changes", first
 * bullet; the rot_in test under "Checks on this head").
 * For each row r and each 128-element block of it:
 *   t[i]  = fp32(x[r][i]) * fp32(suh[i])          (fp32 product, rounded once)
 *   t     = 7 butterfly stages of the 128-point Walsh-Hadamard transform in
 *           fp32, h = 1, 2, ..., 64, pair (p, p+h) with p & h == 0:
 *           lower <- a + b, upper <- a - b
 *   xr[r][i] = fp16_RN(t[i] * 0x1.6a09e6p-4f)     (multiply by the fp32 value
 *           of 1/sqrt(128), then one rounding to fp16)
 * x:   [rows][in_features], dtype x_dtype (TF_F16, TF_BF16 or TF_F32)
 * suh: [in_features] fp16
 * xr:  [rows][in_features] fp16, written
 * rows >= 0 (0 launches nothing); in_features a positive multiple of 128.
 * All pointers 16-byte aligned. Non-finite inputs propagate through their
 * 128-element block.
 */
tf_status tf_rot_in(const void* x, int x_dtype, const void* suh, void* xr,
                    int rows, int in_features, void* stream);

/*
 * tf_trellis_linear -- the trellis-quantized linear for decode rows ("What
 * this changes", second bullet and its sub-bullets):
 *   W[k][n] = mul1(state of the tile weight), decoded inside the kernel from
 *             the packed trellis (format below), never written to memory
 *   acc[r][n] = sum_k xr[r][k] * W[k][n]      (fp16 products, fp32 sums in a
 *             fixed order: a row's bits do not depend on the other rows)
 *   y[r][n] = out( FWHT128(acc[r][block of n])[n] * fp32(1/sqrt(128))
 *                  * fp32(svh[n]) )   (two fp32 multiplies; out() stores the
 *             fp32 value for TF_F32, or rounds it once, to nearest with ties
 *             to even, to fp16 (TF_F16) or bf16 (TF_BF16; "Checks on this
 *             head": the linear at 4 bits with bf16 out); overflow gives
 *             +-inf)
 * xr:      [rows][in_features] fp16 (the output of tf_rot_in)
 * trellis: packed tiles, tf_trellis_bytes(in, out, bits) bytes:
 *   tile (kt, nt), kt < in/16, nt < out/16, is 8*bits uint32 words starting
 *   at word (kt * out/16 + nt) * 8 * bits. Its stream bit j is bit
 *   (31 - j % 32) of word j / 32. Weight i (0..255) of the tile has the
 *   16-bit state made of stream bits ((i+1)*bits - 16 + t) mod (256*bits),
 *   t = 0..15, first bit most significant, and sits at
 *   W[16*kt + i % 16][16*nt + i / 16]. mul1(state): u = state * 0x83DCD12D
 *   mod 2^32, s = sum of u's four bytes, weight = fp16 fma s * 0x1EEE + 0xC2E8
 *   (fp16 bit patterns; 0x1EEE = 0.00676727294921875, 0xC2E8 = -3.453125).
 * svh:     [out_features] fp16
 * y:       [rows][out_features], out_dtype TF_F16, TF_F32 or TF_BF16, written
 * rows >= 0 (0 launches nothing). Rows run in passes of up to 128 on the
 * tcgen05 kernel, each pass
 * decoding the weights once for all its rows ("Known limits": the prompt
 * path, registered bit-equal to this linear): a row's outputs are the same
 * bits whatever pass, slot or batch it runs in, alone or among up to 128
 * rows, because every row goes through the same sequence of per-k-tile
 * tensor-core sums and the same fixed order of partial sums.
 * in/out_features positive multiples of 128;
 * bits in {2, 3, 4, 5, 6, 8}. All pointers 16-byte aligned.
 */
tf_status tf_trellis_linear(const void* xr, const void* trellis, const void* svh,
                            void* y, int out_dtype, int rows, int in_features,
                            int out_features, int bits, void* stream);

/*
 * tf_rot_in_linear -- tf_rot_in followed by tf_trellis_linear in one launch
 * per pass ("What this changes": callers issue rot_in, then the linear, for
 * each projection of a decode step; here the pair is one call). Arguments
 * as in those two calls: x [rows][in_features] of dtype x_dtype, suh
 * [in_features] fp16, xr [rows][in_features] fp16 (written: the rotated
 * rows, the caller's memory), trellis in the k-tile-major order, svh, y,
 * out_dtype, rows, in_features, out_features, bits. xr and y are the same
 * bits as tf_rot_in then tf_trellis_linear give.
 * Inside the launch, the CTAs that are running hand the pass's (row,
 * 128-block) units out among themselves through a counter and rotate them
 * into xr; each CTA's tensor copies of xr start once every unit is written.
 * No CTA waits for another to be resident: one running CTA rotates every
 * unit if it is alone. The wait is bounded like every wait in the kernels
 * (1 s); past it the launch gives up and tf_device_error reports
 * TF_ERR_TIMEOUT. The launch uses three counters of the library's
 * per-device workspace (back at zero after each launch), so, like
 * tf_trellis_linear, it must not run concurrently with another linear call
 * on the same device.
 * Refusals: those of tf_rot_in and tf_trellis_linear.
 */
tf_status tf_rot_in_linear(const void* x, int x_dtype, const void* suh, void* xr,
                           const void* trellis, const void* svh, void* y, int out_dtype,
                           int rows, int in_features, int out_features, int bits,
                           void* stream);

/*
 * tf_rot_in_linear_strips -- tf_rot_in_linear on weights in the strips order
 * of tf_trellis_linear_strips ("Checks on this head": the strips layout); xr
 * and y are the bits of tf_rot_in then tf_trellis_linear_strips. Same
 * arguments, counters and refusals as tf_rot_in_linear.
 */
tf_status tf_rot_in_linear_strips(const void* x, int x_dtype, const void* suh, void* xr,
                                  const void* strips, const void* svh, void* y, int out_dtype,
                                  int rows, int in_features, int out_features, int bits,
                                  void* stream);

/*
 * tf_trellis_linear_strips -- tf_trellis_linear on the same tiles stored in
 * the "strips" order ("Checks on this head": the decode test runs on the
 * checkpoint's tile layout and on the strips layout; the page does not spell
 * that order out, so this one is the library's own). A strip is one block of
 * 128 outputs stored whole. Inside block b < out/128, groups of four k-tiles
 * c < in/64 follow in input order; group c holds the 8 tiles
 * (kt = 4c + kk, nt = 8b + nn) with their words interleaved: word w of tile
 * (4c + kk, 8b + nn) is strips word
 *   (((b * in/64 + c) * 8 + nn) * 8*bits + w) * 4 + kk,   kk < 4, nn < 8.
 * Each unit of work of a block is then one contiguous run, and one 128-bit
 * load brings a word of four k-tiles, which makes the decode cheaper than on
 * the k-tile-major order.
 * Same arguments, results (bit for bit) and refusals as tf_trellis_linear.
 */
tf_status tf_trellis_linear_strips(const void* xr, const void* strips, const void* svh,
                                   void* y, int out_dtype, int rows, int in_features,
                                   int out_features, int bits, void* stream);

/*
 * tf_trellis_to_strips -- repacks tiles from the k-tile-major order of
 * tf_trellis_linear into the strips order of tf_trellis_linear_strips
 * (tf_trellis_bytes(in, out, bits) bytes each; the buffers must not overlap).
 * "Checks on this head" names the two tile layouts the decode runs on; this
 * repack between the library's own readings of them has no counterpart on
 * the pages.
 */
tf_status tf_trellis_to_strips(const void* tiles, void* strips, int in_features,
                               int out_features, int bits, void* stream);

/*
 * tf_trellis_workspace_bytes -- (the pages have no counterpart) bytes of
 * caller workspace tf_trellis_linear_ws
 * needs for this shape on the current device (it depends on the device's SM
 * count: 196,608 bytes of partial sums per SM for passes of up to 128 rows,
 * plus 4 bytes per output block), or 0 for an invalid shape or width, or
 * when no device is usable.
 */
size_t tf_trellis_workspace_bytes(int in_features, int out_features, int bits);

/*
 * tf_trellis_linear_ws -- tf_trellis_linear (layout 0: the k-tile-major
 * tiles) or tf_trellis_linear_strips (layout 1: the strips order) with the
 * scratch in caller memory instead of the library's per-device workspace,
 * so that calls with distinct workspaces may run at the same time on
 * different streams of one device. The pages have no counterpart (they
 * describe one call at a time).
 * workspace: device memory of the current device, 256-byte aligned, at least
 *   tf_trellis_workspace_bytes(in_features, out_features, bits) bytes, owned
 *   by the caller; each call clears the part it counts arrivals in with
 *   cudaMemsetAsync on `stream`, so it needs no initialisation. Calls that
 *   share one workspace must be ordered by the caller.
 * Same results (bit for bit) as the entry points above; refusals as theirs,
 * plus TF_ERR_SHAPE for a layout other than 0 or 1, TF_ERR_NULL / TF_ERR_ALIGN
 * for the workspace, and TF_ERR_SCRATCH when workspace_bytes is too small.
 */
tf_status tf_trellis_linear_ws(const void* xr, const void* trellis, const void* svh,
                               void* y, int out_dtype, int rows, int in_features,
                               int out_features, int bits, int layout, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * tf_trellis_linear_noalloc -- the same computation as tf_trellis_linear
 * (same arguments, layouts and results bit for bit; the same refusals, plus
 * TF_ERR_SCRATCH above 2,097,152 outputs) for callers that must not
 * let a library allocate device memory: for example a serving process whose
 * caching allocator has already reserved the memory it plans around, where
 * a cudaMalloc can fail or break that plan, or code that cannot accept the
 * implicit device synchronisation cudaMalloc and cudaFree may cause. The
 * pages describe no counterpart; this is an addition of this library.
 * Its scratch (partial sums of output blocks shared by two thread blocks and
 * one arrival counter per output block) lives in a fixed device array of
 * about 2.6 MB that every GPU loading this library holds until the process
 * exits. Limits: out_features <= 2,097,152 (16,384 blocks of 128), else
 * TF_ERR_SCRATCH; at most 160 thread blocks per launch. The first call on a
 * device looks up the array's device address on that device (call it once
 * before capturing work into a CUDA graph). Each pass of up to 16 rows first
 * clears the counters it uses with cudaMemsetAsync on `stream` (so a pass
 * that gave up a bounded wait leaves nothing stale for the next). All calls
 * share the one array, so
 * calls whose work overlaps on the GPU (for example on two streams) race and
 * must be ordered by the caller. Calls no cudaMalloc or cudaFree. It runs
 * its passes of up to 16 rows on the mma.sync kernel (whose partial sums fit
 * the array); every output has the same bits as tf_trellis_linear's, which
 * runs its passes on the tcgen05 kernel.
 */
tf_status tf_trellis_linear_noalloc(const void* xr, const void* trellis, const void* svh,
                                    void* y, int out_dtype, int rows, int in_features,
                                    int out_features, int bits, void* stream);

/*
 * tf_trellis_decode -- the weights alone: writes the dense fp16 matrix
 * w[in_features][out_features] that tf_trellis_linear decodes internally
 * (same format and codebook as above; "Checks on this head": the linear
 * decodes every width's weights bit for bit).
 */
tf_status tf_trellis_decode(const void* trellis, void* w, int in_features,
                            int out_features, int bits, void* stream);

/*
 * tf_selftest_stranded_wait -- a self-test of the failure path every kernel
 * of this library has: launches, on `stream`, one tiny kernel whose
 * shared-memory barrier wait is never completed. The wait gives up after the
 * library's bounded-wait limit (1 s of GPU time), records that in the
 * device error flag and returns; the next tf_device_error(stream) returns
 * TF_ERR_TIMEOUT and clears the flag, and the CUDA context stays usable.
 * The pages have no counterpart (their planted faults run on the host).
 * Returns TF_OK when the kernel was launched.
 */
tf_status tf_selftest_stranded_wait(void* stream);

/* Bytes of a packed trellis: in_features * out_features * bits / 8, or 0 for
 * an invalid shape or width. The size follows from the format of "What this
 * changes", second bullet: 16 x 16 tiles, each weight one step of a
 * bits-per-weight trellis, so a tile is 256 * bits bits (the tile layout
 * above), and in/16 * out/16 tiles make the matrix. */
size_t tf_trellis_bytes(int in_features, int out_features, int bits);

/* Static text for a status code. The refusal codes (TF_ERR_SHAPE,
 * TF_ERR_BITS, TF_ERR_DTYPE, TF_ERR_NULL, TF_ERR_ALIGN) play the part of the
 * launches' refusals of shapes they do not fit and of unknown widths ("What
 * this changes", last bullet: the launches with the shapes they refuse); the
 * others (TF_ERR_CUDA, TF_ERR_TIMEOUT, TF_ERR_POINTER, TF_ERR_SCRATCH) are
 * this library's own records, with no counterpart on the pages. */
const char* tf_status_string(int status);

/* Text of the last TF_ERR_CUDA on the calling host thread ("" if none).
 * The pages have no counterpart. */
const char* tf_last_error(void);

/*
 * tf_device_error -- synchronises `stream`, then returns TF_ERR_TIMEOUT if a
 * kernel of this library on the current device gave up a bounded wait since
 * the last call (and clears that record), TF_ERR_CUDA if the synchronisation
 * failed, else TF_OK. The pages have no counterpart (their kernels have no
 * waits that can give up).
 */
tf_status tf_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TF_EXL3_H */
