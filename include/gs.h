/*
 * gs.h -- C ABI of the fused guided denoise step for GB300 (sm_103a).
 *
 * One sampler step of a diffusion model, after the model has produced its
 * outputs for the step: regional conditioning accumulation (positive and, with
 * negative regions, uncond branch), classifier-free guidance with a scalar or
 * bucketized per-sample scale, inpaint blend with the original latent and the
 * Euler or Euler-ancestral update to the next sigma, optionally with the next
 * model input under the inpaint wrapper -- all in one kernel launch.  Host
 * helpers build the sigma schedule and the bucket plan once per run, convert
 * areas to latent slices and pack cond entries into model calls; small kernels
 * prepare the latent inpaint mask and its row summary once per run.
 *
 * Sources (page title, section):
 *   [SAMPLING] "12 · 采样器、调度器与 CFG" -- ComfyUI's sampler / scheduler / CFG notes.
 *   [BCG]      the write-up on Bucketized Continuous Guidance in SGLang
 *              (zwxr.cn news 258547), sections 2-4.
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer.  The library allocates nothing, keeps no
 *     pointer after a call returns and never synchronises the stream.
 *   - Device work is enqueued on the caller's stream (a cudaStream_t passed as
 *     gs_stream; NULL is the legacy default stream).
 *   - Errors are returned as gs_status; nothing is launched when an argument
 *     check fails.  No call aborts, throws or traps.  Errors found on the device
 *     (they depend on device-resident step indices) are OR-ed into an optional
 *     caller-owned status word; gs_status_from_word() decodes it.
 *   - Layouts are dense row-major (NCHW) unless a stride is given.
 */
#ifndef GS_H
#define GS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL = the legacy default stream. */
typedef struct CUstream_st* gs_stream;

typedef enum gs_status {
    GS_OK = 0,
    GS_ERR_INVALID_ARG = 1,   /* a pointer, size, rectangle or option is invalid      */
    GS_ERR_UNSUPPORTED = 2,   /* a valid request the library cannot serve             */
    GS_ERR_CUDA = 3,          /* the CUDA runtime reported an error (launch, device)  */
    GS_ERR_STEP_RANGE = 4,    /* device: a step index did not address sigma[i], sigma[i+1]
                                 (or the scale table); that sample was skipped        */
    GS_ERR_NEED_UNCOND = 5,   /* device: a sample's scale was not 1 but no uncond
                                 branch was given; that sample was skipped            */
    GS_ERR_SIGMA = 6,         /* device: sigma[i] <= 0 or not finite; sample skipped */
    GS_ERR_CAPACITY = 7,      /* output buffer too small                              */
    GS_ERR_TIMEOUT = 8        /* device: a pipeline wait gave up (200 ms); the step's
                                 output is incomplete                                 */
} gs_status;

/* Bits of the device status word (uint32, caller-owned, zeroed by the caller). */
#define GS_DEV_STEP_RANGE  1u
#define GS_DEV_NEED_UNCOND 2u
#define GS_DEV_SIGMA       4u
#define GS_DEV_TIMEOUT     8u

/* Storage types of latents and model outputs; arithmetic is always fp32. */
enum { GS_DTYPE_F32 = 0, GS_DTYPE_BF16 = 1, GS_DTYPE_F16 = 2 };

/* Largest number of regional conditioning entries one step accepts. */
#define GS_MAX_REGIONS 16

/* ------------------------------------------------------------------------ */
/* Sigma schedule (host).                                                    */
/* ------------------------------------------------------------------------ */

enum { GS_SCHED_KARRAS = 0, GS_SCHED_NORMAL = 1 };

typedef struct gs_schedule_desc {
    int32_t kind;               /* GS_SCHED_KARRAS or GS_SCHED_NORMAL                   */
    int32_t steps;              /* steps to take, >= 1                                   */
    double  sigma_min;          /* Karras only: lowest nonzero sigma, > 0                */
    double  sigma_max;          /* Karras only: highest sigma, > sigma_min               */
    double  rho;                /* Karras only: exponent, > 0 (7 is usual)               */
    double  denoise;            /* (0, 1): tail of a longer schedule; >= 1: full         */
    int32_t start_step;         /* -1 = none; else drop sigmas before this index         */
    int32_t last_step;          /* -1 = none; else keep sigmas up to this index          */
    int32_t force_full_denoise; /* nonzero: the final sigma is set to 0                  */
    int32_t n_train;            /* normal only: discrete table length (1000)             */
    double  beta_start;         /* normal only: first beta (0.00085)                     */
    double  beta_end;           /* normal only: last beta (0.012)                        */
} gs_schedule_desc;

/*
 * gs_sigmas -- the 1-D sigma sequence a sampler walks, high to low.
 *
 * [SAMPLING] "sigma 序列": built from the model's sampling parameters and the
 * scheduler's name; "denoise 小于 1": a longer base schedule is built and only
 * its tail kept, then start_step / last_step crop it; "force_full_denoise": the
 * final sigma is forced to 0.
 *   Karras: Karras et al. 2022 eq. (5), steps levels evenly spaced in
 *           sigma^(1/rho) from sigma_max to sigma_min, then 0.
 *   normal: the Stable Diffusion scaled-linear discrete table (n_train betas,
 *           sqrt-linear from beta_start to beta_end, sigma_k =
 *           sqrt((1 - abar_k)/abar_k)), sampled from its last entry to its first
 *           at evenly spaced fractional indices with log-linear interpolation,
 *           then 0.
 *   Order: base (int(steps/denoise) steps when denoise < 1, keeping the last
 *   steps+1 values), last_step crop, start_step crop (a start at or past the
 *   last step leaves an empty schedule), force_full_denoise.
 * All arithmetic is binary64; values are rounded to fp32 on output.
 *
 * out:             host float[cap]; receives *n_out values.
 * n_out:           host; number of sigmas written (0 = nothing left to do).
 * base_offset_out: host, may be NULL; index of out[0] in the base schedule.
 * Errors: GS_ERR_INVALID_ARG (NULL desc/out/n_out, steps < 1, denoise <= 0,
 *         bad Karras parameters, kind unknown), GS_ERR_CAPACITY (cap too small;
 *         *n_out still receives the needed length).
 */
gs_status gs_sigmas(const gs_schedule_desc* desc, float* out, int32_t cap,
                    int32_t* n_out, int32_t* base_offset_out);

/* ------------------------------------------------------------------------ */
/* Bucket plan (host).                                                       */
/* ------------------------------------------------------------------------ */

enum { GS_CURVE_LINEAR = 0, GS_CURVE_STEP = 1, GS_CURVE_TABLE = 2, GS_CURVE_PEAK = 3 };

typedef struct gs_curve_desc {
    int32_t kind;   /* GS_CURVE_LINEAR: v0 at progress 0 -> v1 at progress 1
                       GS_CURVE_STEP:   v0 while progress < edge, v1 afterwards
                                        ([BCG] section 5 "front high, then flat")
                       GS_CURVE_PEAK:   v1 at progress 0 and 1, rising linearly to v0 at
                                        progress edge, 0 < edge < 1 ([BCG] section 5
                                        "middle peak")
                       GS_CURVE_TABLE:  the table argument gives one scale per bucket */
    double  v0;
    double  v1;
    double  edge;
    int32_t interp; /* 0: a bucket's scale is the curve at its midpoint progress;
                       1: "simple linear interpolation" inside a bucket ([BCG] section
                       2): a step's scale is the straight line between the curve's
                       values at its bucket's edges b/N and (b+1)/N, at the step's
                       progress.  Not with GS_CURVE_TABLE. */
} gs_curve_desc;

/*
 * gs_bucket_plan -- per-step bucket ids and guidance scales.
 *
 * [BCG] section 2: progress = step / steps, bucket = min(int(progress *
 * num_buckets), num_buckets - 1), evaluated in binary64 as written; the curve
 * is cut into num_buckets constant segments.  Section 4 stage 1: each step
 * reads its scale from the per-bucket table.  A bucket's scale is the curve at
 * the bucket's midpoint progress (b + 1/2)/num_buckets, unless an explicit
 * table is given or curve->interp asks for interpolation inside the bucket
 * (then step i's scale is c(b/N) + (c((b+1)/N) - c(b/N)) * (i/steps * N - b)).
 *
 * steps:           the schedule's step count (n_sigmas - 1), >= 1.
 * num_buckets:     >= 1.
 * curve:           host; see gs_curve_desc.
 * table:           host double[num_buckets] for GS_CURVE_TABLE, else ignored.
 * bucket_of_step:  host int32[steps], may be NULL.
 * scale_of_step:   host float[steps] (the scale LUT the step kernel reads),
 *                  may be NULL.
 * Errors: GS_ERR_INVALID_ARG (also: interp with a table, a peak apex outside (0, 1)).
 */
gs_status gs_bucket_plan(int32_t steps, int32_t num_buckets, const gs_curve_desc* curve,
                         const double* table, int32_t* bucket_of_step, float* scale_of_step);

/* ------------------------------------------------------------------------ */
/* Inpaint mask preparation (device, once per run).                          */
/* ------------------------------------------------------------------------ */

/*
 * gs_mask_prepare -- pixel mask -> latent mask.
 *
 * [SAMPLING] "inpaint 与 mask": the mask is reshaped and interpolated to the
 * latent size (the channel broadcast happens inside gs_guided_step).  Bilinear
 * with half-pixel centres (align_corners = False): destination j samples the
 * source at (j + 1/2) * in/out - 1/2, clamped at 0, upper neighbour clamped to
 * the last pixel.  Index and weight arithmetic is binary64 per pixel; the
 * result is rounded to fp32.
 *
 * pix_mask: device float[B][1][Hp][Wp].   lat_mask: device float[B][1][H][W].
 * Errors: GS_ERR_INVALID_ARG (NULL pointers, sizes < 1), GS_ERR_CUDA.
 */
gs_status gs_mask_prepare(const float* pix_mask, int32_t B, int32_t Hp, int32_t Wp,
                          float* lat_mask, int32_t H, int32_t W, gs_stream stream);

/*
 * gs_mask_rows -- which rows of a latent mask carry any nonzero value.
 *
 * Where a sample's mask is 0 on a whole row, the inpaint blend keeps the original
 * there (den = 0 * pred + 1 * original, [SAMPLING] "inpaint 与 mask"), so the guided
 * prediction of that row is not needed.  This summary, computed once per run,
 * lets gs_guided_step skip reading it (gs_step_args.mask_rows).
 *
 * lat_mask: device float[Bm][1][H][W] (row pitch W).
 * rows_out: device uint32[Bm][ceil(H/32)]: bit (y mod 32) of word y/32 of mask b
 *           is 1 when some lat_mask[b][0][y][x] != 0 (NaN counts as nonzero,
 *           -0 as zero).  Caller-owned.
 * Errors: GS_ERR_INVALID_ARG (NULL pointers, sizes < 1), GS_ERR_CUDA.
 */
gs_status gs_mask_rows(const float* lat_mask, int32_t Bm, int32_t H, int32_t W,
                       uint32_t* rows_out, gs_stream stream);

/*
 * gs_mask_spans -- the nonzero column span of every row of a latent mask.
 *
 * Where a sample's mask is 0, the inpaint blend keeps the original (den = 0 * pred
 * + 1 * original, [SAMPLING] "inpaint 与 mask"), so the guided prediction there is
 * not needed.  This summary, computed once per run, lets gs_guided_step skip the
 * prediction reads of whole bands of rows (like gs_mask_rows) and, in the bands it
 * reads, narrow them to the columns between the band's first and last nonzero
 * mask value (gs_step_args.mask_spans).
 *
 * lat_mask:  device float[Bm][1][H][W] (row pitch W), W <= 65535.
 * spans_out: device uint32[Bm][H]: word y of mask b is lo | (hi << 16), lo the first
 *            and hi - 1 the last column x with lat_mask[b][0][y][x] != 0 (NaN counts
 *            as nonzero, -0 as zero); 0 for a row with no nonzero value.
 *            Caller-owned.
 * Errors: GS_ERR_INVALID_ARG (NULL pointers, sizes < 1), GS_ERR_UNSUPPORTED
 *         (Bm or W above 65535), GS_ERR_CUDA.
 */
gs_status gs_mask_spans(const float* lat_mask, int32_t Bm, int32_t H, int32_t W,
                        uint32_t* spans_out, gs_stream stream);

/* ------------------------------------------------------------------------ */
/* The guided step (device, one kernel launch per call).                     */
/* ------------------------------------------------------------------------ */

/*
 * A regional conditioning output ([SAMPLING] "calc_cond_batch()"): the model's
 * output for the latent crop rows y0..y0+h-1, columns x0..x0+w-1, added back
 * into the frame with weight strength * feather * mask.
 *   feather: ramp width F in latent pixels (0 = none).  Every rectangle edge
 *            that is not on the latent border ramps linearly: a pixel at
 *            distance t (0-based) from it gets min(1, (t+1)/F); the factors of
 *            the edges multiply.
 *   mask:    device float[.][h][w] (row pitch w) or NULL (= 1); sample b reads
 *            mask + b * mask_bstride (mask_bstride 0 = one mask for all samples).
 *   out:     device, storage dtype, [B][C][h][pitch], pitch >= w; columns
 *            w..pitch-1 are never read.
 *   t_start, t_end: the region's timestep range ([SAMPLING] "calc_cond_batch()":
 *            each entry first checks whether the current timestep is valid for it):
 *            the region takes part for sample b only when t_start <= i/S < t_end,
 *            i = the sample's step index, S = n_sigmas - 1, evaluated in binary64
 *            (the progress the guidance buckets use).  t_end <= t_start (a zeroed
 *            struct) means no range: every step.  The TMA-fed kernels do not read
 *            a region's output for the samples whose step is out of its range
 *            (except with negative regions).
 *   negative: 0 = the region is part of the positive (cond) branch; 1 = of the
 *            uncond branch (regional uncond: negative conditioning carries the same
 *            area, mask and strength metadata, [SAMPLING] "negative 不是简单“反向
 *            prompt”").  Each branch is the weight-normalised sum of its entries:
 *            the full-frame output (cond or uncond, weight 1, if given) and its
 *            regions; a pixel no entry of a branch covers gets 0 in that branch.
 *            The positive branch needs cond or a positive region.  Other values are
 *            GS_ERR_INVALID_ARG.
 */
typedef struct gs_region {
    int32_t     y0, x0, h, w;
    float       strength;
    int32_t     feather;
    const float* mask;
    int64_t     mask_bstride;
    const void* out;
    int64_t     pitch;
    double      t_start, t_end;
    int32_t     negative;
} gs_region;

/* samplers (gs_step_args.sampler) */
enum { GS_SAMPLER_EULER = 0, GS_SAMPLER_EULER_ANCESTRAL = 1 };

/* launch_flags */
#define GS_LAUNCH_PDL    1u  /* launch with programmatic dependent launch: the kernel
                                may be scheduled before the previous kernel in the
                                stream ends; it waits for it before it reads or writes
                                any argument's memory (the TMA kernel asks L2 for the
                                lines of its input boxes before the wait, a cache hint
                                that reads no value)                                  */
#define GS_LAUNCH_NO_TMA 2u  /* use the register-streaming kernel even where the
                                TMA-pipelined one applies (same results)            */
#define GS_LAUNCH_TEST_WAIT_TIMEOUT 4u
                             /* tests of the error path only: every tile of the TMA
                                kernel also waits for 16 bytes that never arrive, so
                                its bounded wait (200 ms) expires; the kernel then
                                sets GS_DEV_TIMEOUT and writes no output.  All real
                                transfers still complete before any CTA exits.      */

typedef struct gs_step_args {
    int32_t B, C, H, W;         /* latent batch, channels, rows, columns (all >= 1)      */
    int32_t dtype;              /* GS_DTYPE_*: storage type of every latent-shaped buffer */

    const void* x;              /* device [B][C][H][W]: the current latent x_i           */
    void*       x_out;          /* device [B][C][H][W]: x_{i+1}; may alias x             */
    void*       denoised_out;   /* device [B][C][H][W] or NULL: the blended prediction   */

    /* Model outputs of this step.  A stacked [2B][C][H][W] output laid out as
       [uncond_0 .. uncond_{B-1}, cond_0 .. cond_{B-1}] ([BCG] section 3) is passed
       as uncond = base, cond = base + B*C*H*W elements. */
    const void* uncond;         /* device [B][C][H][W], or NULL when the uncond forward
                                   was skipped because every scale is 1 ([SAMPLING]
                                   "cfg = 1 的优化")                                   */
    const void* cond;           /* device [B][C][H][W], or NULL when regions give the
                                   positive branch.  With regions it joins them as a
                                   full-frame entry of weight 1.                        */
    int32_t n_regions;          /* 0 .. GS_MAX_REGIONS                                   */
    const gs_region* regions;   /* host array[n_regions]                                 */

    /* Schedule and guidance. */
    const float*   sigmas;      /* device float[n_sigmas], high to low                   */
    int32_t        n_sigmas;    /* >= 2                                                  */
    const int32_t* step_idx;    /* device int32[B]: sample b steps from sigmas[i] to
                                   sigmas[i+1], i = step_idx[b]; NULL = every sample
                                   takes `step`                                          */
    int32_t        step;        /* used when step_idx is NULL: 0 <= step <= n_sigmas-2   */
    const float*   scale_lut;   /* device float[n_lut]: scale of sample b is
                                   scale_lut[i]; NULL = `cfg` for every sample           */
    int32_t        n_lut;
    float          cfg;

    /* Inpaint ([SAMPLING] "inpaint 与 mask"): den = m*pred + (1-m)*original with the
       latent mask m broadcast over channels (1 = regenerate, 0 = keep original). */
    const float*   inpaint_mask;   /* device float[.][1][H][W] or NULL (no inpaint)      */
    int64_t        mask_bstride;   /* elements between samples' masks; 0 = shared        */
    const uint8_t* mask_present;   /* device uint8[B] or NULL (= every sample); samples
                                      with 0 are not blended and their mask and
                                      original are not read                             */
    const void*    original;       /* device [B][C][H][W]; required with inpaint_mask    */

    uint32_t* dev_status;       /* device uint32 or NULL: GS_DEV_* bits OR-ed in         */
    uint32_t  launch_flags;     /* GS_LAUNCH_*                                           */

    /* Optional row summary of inpaint_mask from gs_mask_rows: device
       uint32[.][ceil(H/32)], one row of words per mask, sample b's at
       b * ceil(H/32) words (0 when mask_bstride is 0); NULL = not given.  Given it,
       the TMA-fed kernels read neither uncond, cond nor any region output for a
       band of rows in which a blended sample's mask is 0 on every row: there
       den = original exactly, whatever the prediction (the prediction is taken as
       0, so a non-finite prediction there does not propagate).  The caller keeps
       it in step with inpaint_mask. */
    const uint32_t* mask_rows;

    /* Sampler ([SAMPLING] "sampler_object": names map onto k-diffusion functions).
       GS_SAMPLER_EULER (0, default): x' = den + (sigma_next/sigma) (x - den).
       GS_SAMPLER_EULER_ANCESTRAL (1, eta = 1): x' = den + (sigma_down/sigma) (x - den)
       + sigma_up * noise, sigma_up = min(sigma_next, sqrt(sigma_next^2 (sigma^2 -
       sigma_next^2) / sigma^2)), sigma_down = sqrt(sigma_next^2 - sigma_up^2), per sample
       in fp32.  Needs `noise`.  A sample whose sigma_next is negative (or NaN) has no
       split: it is flagged GS_DEV_SIGMA and left unwritten, like sigma <= 0.
       Any other value of `sampler` is GS_ERR_INVALID_ARG. */
    int32_t     sampler;
    const void* noise;          /* device [B][C][H][W], storage dtype: this step's fresh
                                   noise (the random numbers are an input)              */
    /* Optional second output under the inpaint wrapper ([SAMPLING] "inpaint 与 mask":
       each step the unmasked region is replaced by the original, the noise kept to the
       mask): the next model call's input m * x' + (1 - m) * (original + sigma_next *
       orig_noise), x' for samples without a mask.  Needs inpaint_mask, original and
       orig_noise.  It may alias x (each element is read before it is written) but must
       not overlap x_out or denoised_out (the same start address is GS_ERR_INVALID_ARG). */
    void*       model_in_out;   /* device [B][C][H][W] or NULL                           */
    const void* orig_noise;     /* device [B][C][H][W]: the run's fixed noise            */

    /* Optional span summary of inpaint_mask from gs_mask_spans: device uint32[.][H],
       sample b's rows at b * H words (0 when mask_bstride is 0); NULL = not given.  It
       takes the place of mask_rows (which is then ignored): the TMA-fed kernels skip
       the prediction reads of a blended band whose mask is 0 on every row, as with
       mask_rows, and in the other bands of a blended sample read uncond and cond
       only from the band's first to its last nonzero mask column (rounded out to
       16-byte vectors; loaded as 128-byte column chunks aligned to 128 bytes of the
       row, DRAM's unit of transfer to L2, or as whole rows): outside that span the
       prediction is taken as 0 (den is the original exactly there, up to the sign of
       zero), so a non-finite prediction there does not propagate.  Region outputs
       are read whole in the bands they touch.
       The caller keeps it in step with inpaint_mask.  Negative regions: ignored. */
    const uint32_t* mask_spans;
    /* 0 or 1.  With 1, a sample whose scale is exactly 1 does not read its uncond
       output in the TMA-fed kernels: pred = pos exactly, the per-sample form of
       [SAMPLING] "cfg = 1 的优化" (the uncond branch is still given for the other
       samples).  The uncond box of every sample then waits for the sample's scale
       (two dependent loads), so set it only when the scale table holds a 1 (or cfg
       is 1).  Negative regions: ignored.  Other values: GS_ERR_INVALID_ARG. */
    int32_t     unit_scale_skip;
} gs_step_args;

/*
 * gs_guided_step -- one guided denoise step for every sample of the batch.
 *
 * For sample b with i = step_idx[b], sigma = sigmas[i], sigma_next =
 * sigmas[i+1], s = scale_lut[i] (or cfg), all arithmetic in fp32:
 *   pos  = cond                                  (no regions), or
 *          sum_r w_r*out_r / sum_r w_r           ([SAMPLING] calc_cond_batch:
 *                                                 accumulate by strength and mask,
 *                                                 normalise overlaps by summed
 *                                                 weight; 0 where no entry covers;
 *                                                 the division multiplies by the
 *                                                 hardware reciprocal, relative
 *                                                 error below 2^-22, exact for a
 *                                                 summed weight of 1)
 *   pred = fma(s, pos, (1-s)*uncond)             ([SAMPLING] "CFG 的核心", [BCG]
 *                                                 sections 3-4: uncond +
 *                                                 s*(cond-uncond) in fp32, exact
 *                                                 at s = 0 and s = 1); pred = pos
 *                                                 when uncond is NULL
 *   den  = fma(m, pred, (1-m)*original)          (inpaint samples), else pred
 *   x'   = fma(sigma_next/sigma, x - den, den)   (Euler: x + (sigma_next-sigma)*
 *                                                 (x-den)/sigma; exact den at
 *                                                 sigma_next = 0)
 * rounded to the storage dtype (round to nearest even).
 *
 * Samples whose step index is out of range, whose sigma is not positive, or
 * that need the missing uncond branch are skipped (x_out and denoised_out are
 * not written for them) and flagged in dev_status.
 *
 * Kernels (all give the same results):
 *   - TMA-pipelined: used when every latent-shaped pointer is 16-byte aligned,
 *     W * element size is a multiple of 16 bytes, every region output is 16-byte
 *     aligned with a 16-byte-multiple row pitch, and the inpaint mask is
 *     per-sample dense or shared.  Tensor maps are encoded per call (about a
 *     microsecond of host time; gs_step_prepare does it once).  One CTA per
 *     tile of (sample, up to 4 channels, a band of rows, whole rows or a block
 *     of columns: rows wider than 256 columns, or whose 16-byte groups make no
 *     whole warps, are cut into blocks); the channels and band height of a
 *     tile follow the step's size and options (64 to 256 threads a tile; a tile
 *     whose stage would not fit a CTA's shared memory takes fewer rows, then
 *     fewer channels), or are set with the environment variables
 *     GS_TMA_CHANNELS and GS_TMA_ROWS (tuning knobs; results do not change).
 *     Each tile asks L2 for the lines of its x and prediction boxes before it
 *     waits for the previous kernel (see GS_LAUNCH_PDL).
 *   - register-streaming with 16-byte vectors: pointers 16-byte aligned and W a
 *     multiple of 16 bytes / element size; one item of 8 (16-bit) or 4 (fp32)
 *     pixels x 2 channels per thread, or as many channels (1, 2 or 4) as the
 *     environment variable GS_STEP_CHANNELS asks (a tuning knob);
 *   - scalar: anything else.
 * x_out may alias x (or another latent-shaped input); it must not overlap
 * region outputs or masks.
 *
 * Errors: GS_ERR_INVALID_ARG (NULL required pointer, size < 1, region outside
 * the frame or pitch < w, n_regions out of range, step out of range with
 * step_idx NULL, neither cond nor a positive region, a negative flag other than
 * 0 / 1, inpaint without original, unknown dtype or sampler, the ancestral
 * sampler without noise, the model input without inpaint_mask or orig_noise or
 * on x_out / denoised_out, mask_rows or mask_spans without inpaint_mask or not
 * 4-byte aligned, mask_spans with W above 65535, unit_scale_skip not 0 or 1),
 * GS_ERR_CUDA (launch failure).  Device-found errors: see dev_status.
 */
gs_status gs_guided_step(const gs_step_args* args, gs_stream stream);

/* ---- Prepared launches ------------------------------------------------------------
 * A sampler that steps the same buffers many times can check the arguments and build
 * the launch once (gs_step_prepare) and then launch one step per call
 * (gs_step_launch), which skips the argument checks and the tensor-map encoding
 * gs_guided_step repeats on every call.  The plan is caller-owned host memory; the
 * library allocates nothing.  The plan holds the device pointers of the arguments it
 * was prepared from: the caller keeps those buffers alive and unmoved while it uses
 * the plan, and prepares a new plan for other buffers (e.g. one plan per buffer of a
 * ping-pong pair).  The step's results are those of gs_guided_step with the same
 * arguments ([SAMPLING] "comfy.sample.sample()": the sampler calls the same step
 * function every step; only the step index moves).
 */
#define GS_STEP_PLAN_BYTES 8192
typedef struct gs_step_plan {
    uint64_t opaque[GS_STEP_PLAN_BYTES / 8];   /* any 8-byte-aligned host memory */
} gs_step_plan;

/*
 * gs_step_prepare -- check the arguments as gs_guided_step does and write a plan.
 * args: as for gs_guided_step (args->step is ignored: gs_step_launch passes it);
 * plan: host, caller-owned, written in full.
 * Errors: those of gs_guided_step's checks; GS_ERR_INVALID_ARG for a NULL plan.
 */
gs_status gs_step_prepare(const gs_step_args* args, gs_step_plan* plan);

/*
 * gs_step_launch -- one step from a plan, enqueued on `stream` (one kernel launch).
 * step: the step index of every sample (0 <= step <= n_sigmas - 2) when the plan was
 *       prepared without step_idx; ignored otherwise.
 * Errors: GS_ERR_INVALID_ARG (NULL or unprepared plan, step out of range),
 *         GS_ERR_CUDA (launch failure).  Device-found errors: see dev_status.
 */
gs_status gs_step_launch(const gs_step_plan* plan, int32_t step, gs_stream stream);

/* Kernels gs_guided_step chooses between (same results, different data movement). */
enum { GS_KERNEL_SCALAR = 0, GS_KERNEL_VECTOR = 1, GS_KERNEL_TMA = 2 };

/*
 * gs_step_kernel_kind -- which kernel gs_guided_step would launch for these
 * arguments, after the same argument checks, without launching anything.
 * kind: host int32; receives GS_KERNEL_*.  Errors: as gs_guided_step's checks.
 */
gs_status gs_step_kernel_kind(const gs_step_args* args, int32_t* kind);

/* ---- Host helpers of the conditioning pass ------------------------------------
 * [SAMPLING] "calc_cond_batch()": for each conditioning entry the pass turns its
 * area (a percentage or coordinates) into a latent slice, and decides which entries
 * can share one model call and how many to merge given the free memory; "为什么要
 * 自己拼 batch": cond, uncond and regions batch together when shape and control
 * options agree, and are split when memory runs short.  Both helpers are plain host
 * code (no device memory, no stream).
 */
enum { GS_AREA_LATENT = 0, GS_AREA_PIXELS = 1, GS_AREA_FRACTION = 2 };

typedef struct gs_area {
    int32_t units;          /* GS_AREA_*: latent pixels, image pixels or fractions of H, W */
    double  y0, x0, h, w;   /* top-left corner and size in those units                     */
} gs_area;

typedef struct gs_rect {
    int32_t y0, x0, h, w;   /* a latent slice: rows y0 .. y0+h-1, columns x0 .. x0+w-1     */
} gs_rect;

/*
 * gs_areas_to_latent -- for each of n areas, the smallest whole-pixel slice of an
 * H x W latent that covers it, clipped to the frame.  In latent units (image pixels
 * divided by `scale`, the VAE's downscale factor; fractions multiplied by H or W) the
 * area covers [y0, y0+h) x [x0, x0+w); its slice is rows floor(y0) .. ceil(y0+h)-1 and
 * columns floor(x0) .. ceil(x0+w)-1, in binary64.  An area that covers no latent
 * pixel (outside the frame, or of zero height or width) gives h = w = 0 and
 * y0 = x0 = 0; drop it before building gs_region entries.
 * areas: host [n]; out: host [n] (caller-owned).  scale: used for GS_AREA_PIXELS.
 * Errors: n < 0, a NULL array with n > 0, H or W < 1, scale < 1 with a pixel area,
 *         a non-finite corner or size, a negative size, unknown units ->
 *         GS_ERR_INVALID_ARG (out untouched).
 */
gs_status gs_areas_to_latent(const gs_area* areas, int32_t n, int32_t H, int32_t W,
                             int32_t scale, gs_rect* out);

typedef struct gs_cond_entry {
    int32_t h, w;           /* the entry's latent shape (its model input's spatial size)   */
    int32_t rows;           /* batch rows it needs (samples)                               */
    int64_t options;        /* compatibility key of its control options                    */
} gs_cond_entry;

typedef struct gs_cond_chunk {
    int32_t call;           /* model call index, in the order calls open                   */
    int32_t entry;          /* entry index                                                 */
    int32_t row0, rows;     /* that entry's rows row0 .. row0+rows-1                       */
} gs_cond_chunk;

/*
 * gs_pack_conds -- pack n cond entries into model calls.  Entries share a call only
 * when (h, w, options) are equal; a call of shape h x w holds at most
 * max(1, floor(budget / (h*w))) rows, budget being the latent pixels per call the free
 * memory allows.  Entries are taken in order: an entry's rows fill the last call opened
 * for its key while it has room, then new calls of that key, each filled to capacity
 * (so each key uses ceil(its rows / capacity) calls).  Chunks are written entry by
 * entry in row order.
 * entries: host [n]; chunks: host [cap]; *n_chunks, *n_calls: host, receive the counts.
 * Errors: n < 0, NULL arrays, budget < 1, an entry with h, w or rows < 1 ->
 *         GS_ERR_INVALID_ARG; GS_ERR_CAPACITY if more than cap chunks are needed
 *         (*n_chunks then receives the number needed, chunks is partly written).
 */
gs_status gs_pack_conds(const gs_cond_entry* entries, int32_t n, int64_t budget,
                        gs_cond_chunk* chunks, int32_t cap, int32_t* n_chunks,
                        int32_t* n_calls);

/* Decode a device status word into the first gs_status it carries (GS_OK if 0). */
gs_status gs_status_from_word(uint32_t word);

/* A static, human-readable name for a status code. */
const char* gs_status_string(gs_status status);

/* ABI version of this header (bumped on any layout change). */
#define GS_ABI_VERSION 6
int32_t gs_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GS_H */
