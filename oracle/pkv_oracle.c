/*
 * pkv_oracle.c -- reference oracle for the batched paged-KV decode step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the package smoke check and
 * the benchmark's CPU legs (the CPU baseline and the reference arm) load this
 * file's library. The CUDA library
 * never links it, calls it or includes anything from it, and this file includes
 * nothing from the CUDA library.
 *
 * Plain, slow, single-threaded C in fp64 (build with -ffp-contract=off so that
 * every product and sum is rounded exactly as written). Each function cites the
 * passage it follows:
 *
 *  [P2] "手写LLM推理引擎：Tokenizer、Transformer与Detokenizer三段式实现",
 *       section 3.2 (the two RoPE equations and the cos/sin precompute routine,
 *       whose inverse frequency is base^(-2j/dim)).
 *  [P3] "Hours of YouTube and 85 handtyped pages of notes on LLM Inference –
 *       Start here" (the samir-vllm README), feature list: the shared BF16 KV
 *       page pool item (16 tokens of K and V per physical page, block table
 *       per sequence and layer, decode appends the new token at its absolute
 *       RoPE position) and the direct paged decode attention item (each query
 *       head streams its sequence's cached pages, FP32 online softmax).
 *  [P4] "llmc — 从零写一个大模型推理引擎（配套代码）", file table (an explicit
 *       softmax operator) and the introduction (negative return = error).
 *
 * Readings taken where the pages are silent or at odds (all listed in the
 * design notes):
 *  - RoPE pairs dimension j with j + D/2 ("rotate-half"), not (2j, 2j+1) as
 *    [P2]'s equations print them; the workload statement fixes rotate-half.
 *    No frequency scaling: inv_freq_j = theta^(-2j/D) exactly as [P2].
 *  - The rotated key is computed in fp64 (two rounded products, one rounded
 *    sum) and rounded once, to nearest-even, from double to bf16. V is copied.
 *  - The rotated query is kept in fp64 (the GPU keeps fp32); it is not
 *    rounded to bf16.
 *  - Query head i reads KV head i / (Hq/Hkv) (consecutive groups).
 *  - The attention is the plain definition: gather, scores, explicit
 *    two-pass softmax, weighted sum of V. The online form of [P3] computes the
 *    same value up to rounding order.
 *
 * Pool layout (the library's documented contract; the oracle indexes it with
 * its own function): element (page, kv head h, kind K=0/V=1, slot s, dim d)
 * lives at bf16 offset ((((page*Hkv + h)*2 + kind)*P + s)*D + d).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_DIM 256

/* bf16 bits -> double. A bf16 value is the top half of a binary32 value, and
 * every binary32 value is exact in double. */
double oracle_bf16_to_double(uint16_t bits)
{
	uint32_t u = (uint32_t)bits << 16;
	float f;
	memcpy(&f, &u, sizeof f);
	return (double)f;
}

/* double -> bf16, round to nearest, ties to even, from the format's
 * definition: sign, 8 exponent bits (bias 127), 7 fraction bits; below 2^-126
 * the grid is the subnormal grid of spacing 2^-133. The value is scaled so that
 * one unit in the last place is 1, rounded to an integer (ties to even), and
 * scaled back; the result has at most 8 significant bits and is therefore
 * exact in binary32, whose upper half is the bf16 encoding. NaN maps to the
 * canonical quiet NaN 0x7FC0. */
uint16_t oracle_bf16_from_double(double x)
{
	if (isnan(x))
		return 0x7FC0;
	uint16_t sign = signbit(x) ? 0x8000 : 0;
	double a = fabs(x);
	if (isinf(a))
		return sign | 0x7F80;
	if (a == 0.0)
		return sign;
	int e;
	frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1): floor(log2 a) = e - 1 */
	int binade = e - 1;
	if (binade < -126)
		binade = -126;         /* subnormals share the spacing of the lowest binade */
	int ulp_exp = binade - 7;  /* 7 fraction bits */
	double n = nearbyint(ldexp(a, -ulp_exp)); /* exact scaling; default mode: ties to even */
	double r = ldexp(n, ulp_exp);
	if (r >= 0x1p128)
		return sign | 0x7F80;  /* rounds past the largest finite bf16 */
	float f = (float)r;        /* exact */
	uint32_t u;
	memcpy(&u, &f, sizeof u);
	return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

void oracle_bf16_from_double_array(const double *x, uint16_t *out, long n)
{
	for (long i = 0; i < n; i++)
		out[i] = oracle_bf16_from_double(x[i]);
}

/*
 * cos and sin of an fp64 angle, correctly rounded to fp64: the fp64 numbers
 * nearest to the true values. [P2] section 3.2 rotates by cos and sin of the
 * angle m theta_j; the stored key is the bf16 rounding of an fp64 rotation by
 * them, so they are fixed by this definition rather than by whichever math
 * library is linked.
 *
 * Method, in double-double arithmetic (a value is hi + lo, about 106 bits):
 *  - reduction: k = nearest integer to a * 2/pi, r = a - k pi/2 with pi/2 as
 *    the sum of four doubles (each the double nearest to what the previous
 *    ones leave over, pi/2 to about 2^-216), every product k * part exact
 *    (two-product by FMA), the differences summed in double-double;
 *  - Taylor series at |r| <= pi/4 (plus a few ulps), nested:
 *    sin r = r (1 - r^2/(2*3) (1 - r^2/(4*5) (...))),
 *    cos r = 1 - r^2/(1*2) (1 - r^2/(3*4) (...)), 16 factors each, every
 *    step in double-double (division by the integer (2n)(2n+1) or
 *    (2n-1)(2n) done in double-double);
 *  - quadrant k mod 4 picks +-sin r / +-cos r;
 *  - rounding test: the double-double result is within 2^-92 of the true
 *    value relative (plus k 2^-130 absolute for the reduction); if a midpoint
 *    between neighbouring doubles lies that close, the rounding cannot be
 *    decided and the function returns -1 (0 otherwise).
 */
typedef struct {
	double hi, lo;
} ddouble;

static ddouble dd_sum(double a, double b)  /* a + b exactly (Knuth) */
{
	double s = a + b;
	double bb = s - a;
	double e = (a - (s - bb)) + (b - bb);
	ddouble r = { s, e };
	return r;
}

static ddouble dd_quick(double a, double b)  /* a + b exactly, |a| >= |b| (Dekker) */
{
	double s = a + b;
	ddouble r = { s, b - (s - a) };
	return r;
}

static ddouble dd_prod(double a, double b)  /* a * b exactly */
{
	double p = a * b;
	ddouble r = { p, fma(a, b, -p) };
	return r;
}

static ddouble dd_plus(ddouble x, ddouble y)
{
	ddouble s = dd_sum(x.hi, y.hi);
	ddouble t = dd_sum(x.lo, y.lo);
	s = dd_quick(s.hi, s.lo + t.hi);
	return dd_quick(s.hi, s.lo + t.lo);
}

static ddouble dd_times(ddouble x, ddouble y)
{
	ddouble p = dd_prod(x.hi, y.hi);
	return dd_quick(p.hi, p.lo + (x.hi * y.lo + x.lo * y.hi));
}

static ddouble dd_over(ddouble x, double d)  /* x / d */
{
	double q1 = x.hi / d;
	ddouble p = dd_prod(q1, d);
	double rem = ((x.hi - p.hi) - p.lo) + x.lo;
	return dd_quick(q1, rem / d);
}

/* 1 - x, for |x| < 1 */
static ddouble dd_one_minus(ddouble x)
{
	ddouble s = dd_sum(1.0, -x.hi);
	return dd_quick(s.hi, s.lo - x.lo);
}

/* Whether x.hi is the double nearest to every real within eps of x. */
static int dd_decided(ddouble x, double eps)
{
	if (x.hi == 0.0)
		return x.lo == 0.0 && eps == 0.0;
	int e;
	frexp(x.hi, &e);                 /* |x.hi| in [2^(e-1), 2^e) */
	double ulp = ldexp(1.0, e - 53);
	double m = fabs(x.hi);
	int inward = (x.lo < 0.0) == (x.hi > 0.0);
	double half = (inward && m == ldexp(1.0, e - 1)) ? ulp / 4 : ulp / 2;
	return fabs(x.lo) + eps < half;
}

int oracle_cos_sin(double a, double *c, double *s)
{
	static const double pio2[4] = {
		0x1.921fb54442d18p+0, 0x1.1a62633145c07p-54,
		-0x1.f1976b7ed8fbcp-110, 0x1.4cf98e804177dp-164,
	};
	if (!isfinite(a) || fabs(a) >= 0x1p52) {
		*c = *s = NAN;
		return -2;
	}
	int neg = signbit(a) != 0;
	double x = fabs(a);
	double k = nearbyint(x * 0x1.45f306dc9c883p-1);  /* 2/pi rounded */
	ddouble r = { x, 0.0 };
	for (int i = 0; i < 4; i++) {
		ddouble p = dd_prod(k, pio2[i]);
		p.hi = -p.hi;
		p.lo = -p.lo;
		r = dd_plus(r, p);
	}
	ddouble z = dd_times(r, r);
	ddouble ts = { 1.0, 0.0 }, tc = { 1.0, 0.0 };
	for (int n = 16; n >= 1; n--) {
		ts = dd_one_minus(dd_over(dd_times(z, ts), (double)((2 * n) * (2 * n + 1))));
		tc = dd_one_minus(dd_over(dd_times(z, tc), (double)((2 * n - 1) * (2 * n))));
	}
	ddouble sr = dd_times(r, ts), cr = tc;
	ddouble cv, sv;
	switch ((long long)k & 3) {
	case 0: cv = cr; sv = sr; break;
	case 1: cv = sr; cv.hi = -cv.hi; cv.lo = -cv.lo; sv = cr; break;
	case 2: cv = cr; cv.hi = -cv.hi; cv.lo = -cv.lo; sv = sr; sv.hi = -sv.hi; sv.lo = -sv.lo; break;
	default: cv = sr; sv = cr; sv.hi = -sv.hi; sv.lo = -sv.lo; break;
	}
	if (neg) {
		sv.hi = -sv.hi;
		sv.lo = -sv.lo;
	}
	*c = cv.hi;
	*s = sv.hi;
	if (x == 0.0)
		return 0;                    /* cos 0 = 1 and sin 0 = 0 exactly */
	double abs_err = k * 0x1p-130;       /* the reduction is exact when k = 0 */
	int ok = dd_decided(cv, fabs(cv.hi) * 0x1p-92 + abs_err) &&
		 dd_decided(sv, fabs(sv.hi) * 0x1p-92 + abs_err);
	return ok ? 0 : -1;
}

/* [P2] section 3.2, cos/sin precompute: inverse frequency base^(-2j/dim). */
double oracle_rope_inv_freq(double theta, int j, int head_dim)
{
	return pow(theta, -(2.0 * (double)j) / (double)head_dim);
}

/* [P2] section 3.2, the two RoPE equations, read with rotate-half pairing:
 * for j < D/2, with angle = pos * inv_freq_j,
 *   y_j       = x_j * cos - x_{j+D/2} * sin
 *   y_{j+D/2} = x_{j+D/2} * cos + x_j * sin
 * Each product and each sum is one fp64 rounding (no fused multiply-add). */
int oracle_rope_rotate(const double *x, double *y, int head_dim, long pos, double theta)
{
	int half = head_dim / 2;
	int rc = 0;
	for (int j = 0; j < half; j++) {
		double angle = (double)pos * oracle_rope_inv_freq(theta, j, head_dim);
		double c, s;
		if (oracle_cos_sin(angle, &c, &s) != 0)
			rc = -4;             /* cos/sin not decidable: the caller reports it */
		double a = x[j];
		double b = x[j + half];
		double ac = a * c;
		double bs = b * s;
		double bc = b * c;
		double as = a * s;
		y[j] = ac - bs;
		y[j + half] = bc + as;
	}
	return rc;
}

/* Rotate n vectors of length head_dim, vector i at position pos[i]. Returns
 * 0, or -4 when some cos/sin could not be rounded with certainty. */
int oracle_rope_rotate_many(const double *x, double *y, long n, int head_dim,
			    const int32_t *pos, double theta)
{
	int rc = 0;
	for (long i = 0; i < n; i++)
		if (oracle_rope_rotate(x + i * head_dim, y + i * head_dim, head_dim, pos[i], theta))
			rc = -4;
	return rc;
}

/* cos and sin of n angles (oracle_cos_sin); returns the number undecided. */
long oracle_cos_sin_many(const double *a, double *c, double *s, long n)
{
	long bad = 0;
	for (long i = 0; i < n; i++)
		if (oracle_cos_sin(a[i], c + i, s + i) != 0)
			bad++;
	return bad;
}

static size_t pool_offset(long page, int h, int kind, int slot, int d,
			  int num_kv_heads, int head_dim, int page_size)
{
	return ((((size_t)page * num_kv_heads + h) * 2 + kind) * page_size + slot) * head_dim + d;
}

/*
 * [P3] shared page pool item: decode appends the new token at its absolute
 * RoPE position. For sequence b the new token is cache index t = seq_lens[b]-1
 * (seq_lens counts the token), stored in slot t % P of page
 * block_tables[b][t / P]; it is rotated at positions[b].
 *
 * q, k, v are bf16 bits, [B][Hq][D], [B][Hkv][D], [B][Hkv][D]. The rotated
 * query goes to q_rot (fp64, [B][Hq][D]). Returns 0, or -1 for a bad length,
 * -2 for a bad page id, -3 for a bad shape, -4 when a cos/sin could not be
 * rounded with certainty (nothing after the failing sequence is written).
 */
int oracle_append_rope(uint16_t *pool, long num_pages, int num_kv_heads, int head_dim,
		       int page_size, const uint16_t *q, const uint16_t *k, const uint16_t *v,
		       double *q_rot, const int32_t *block_tables, int max_blocks,
		       const int32_t *seq_lens, const int32_t *positions, int batch,
		       int num_q_heads, double theta)
{
	double in[ORACLE_MAX_DIM], out[ORACLE_MAX_DIM];
	if (head_dim <= 0 || head_dim > ORACLE_MAX_DIM || head_dim % 2 || page_size <= 0)
		return -3;
	for (int b = 0; b < batch; b++) {
		int n = seq_lens[b];
		if (n < 1 || n > max_blocks * page_size)
			return -1;
		int t = n - 1;
		long page = block_tables[(size_t)b * max_blocks + t / page_size];
		if (page < 0 || page >= num_pages)
			return -2;
		int slot = t % page_size;
		long pos = positions[b];
		for (int h = 0; h < num_kv_heads; h++) {
			const uint16_t *kh = k + ((size_t)b * num_kv_heads + h) * head_dim;
			const uint16_t *vh = v + ((size_t)b * num_kv_heads + h) * head_dim;
			for (int d = 0; d < head_dim; d++)
				in[d] = oracle_bf16_to_double(kh[d]);
			if (oracle_rope_rotate(in, out, head_dim, pos, theta))
				return -4;
			for (int d = 0; d < head_dim; d++) {
				pool[pool_offset(page, h, 0, slot, d, num_kv_heads, head_dim, page_size)] =
					oracle_bf16_from_double(out[d]);
				pool[pool_offset(page, h, 1, slot, d, num_kv_heads, head_dim, page_size)] = vh[d];
			}
		}
		for (int i = 0; i < num_q_heads; i++) {
			const uint16_t *qh = q + ((size_t)b * num_q_heads + i) * head_dim;
			for (int d = 0; d < head_dim; d++)
				in[d] = oracle_bf16_to_double(qh[d]);
			if (oracle_rope_rotate(in, q_rot + ((size_t)b * num_q_heads + i) * head_dim,
					       head_dim, pos, theta))
				return -4;
		}
	}
	return 0;
}

/* Copy tokens [t0, t1) of (sequence b, kv head h) out of the pool, in logical
 * order, as doubles: K into kd, V into vd ([t1-t0][D] each). */
static int gather(const uint16_t *pool, long num_pages, int num_kv_heads, int head_dim,
		  int page_size, const int32_t *bt_row, int h, int t0, int t1,
		  double *kd, double *vd)
{
	for (int t = t0; t < t1; t++) {
		long page = bt_row[t / page_size];
		if (page < 0 || page >= num_pages)
			return -2;
		int slot = t % page_size;
		for (int d = 0; d < head_dim; d++) {
			kd[(size_t)(t - t0) * head_dim + d] = oracle_bf16_to_double(
				pool[pool_offset(page, h, 0, slot, d, num_kv_heads, head_dim, page_size)]);
			vd[(size_t)(t - t0) * head_dim + d] = oracle_bf16_to_double(
				pool[pool_offset(page, h, 1, slot, d, num_kv_heads, head_dim, page_size)]);
		}
	}
	return 0;
}

/* Attention of one query vector over n gathered tokens with an explicit
 * two-pass softmax ([P4] softmax operator): scores, max, exponentials, sum,
 * weighted sum of V. Also returns the log-sum-exp of the scores. */
static double attend(const double *qv, const double *kd, const double *vd, int n,
		     int head_dim, double scale, double *s, double *o)
{
	double m = -INFINITY;
	for (int t = 0; t < n; t++) {
		double acc = 0.0;
		for (int d = 0; d < head_dim; d++)
			acc += qv[d] * kd[(size_t)t * head_dim + d];
		s[t] = scale * acc;
		if (s[t] > m)
			m = s[t];
	}
	double z = 0.0;
	for (int t = 0; t < n; t++) {
		s[t] = exp(s[t] - m);
		z += s[t];
	}
	for (int d = 0; d < head_dim; d++)
		o[d] = 0.0;
	for (int t = 0; t < n; t++) {
		double p = s[t] / z;
		for (int d = 0; d < head_dim; d++)
			o[d] += p * vd[(size_t)t * head_dim + d];
	}
	return m + log(z);
}

/*
 * [P3] direct paged decode attention item, written as its definition: for
 * every sequence b, every query head i (KV head i / g), attend over the
 * seq_lens[b] tokens the block table maps. q_rot fp64 [B][Hq][D] -> out fp64
 * [B][Hq][D]. Returns 0, -1 bad length, -2 bad page id, -3 bad shape, -4 no
 * memory.
 */
int oracle_gqa_decode(const uint16_t *pool, long num_pages, int num_kv_heads, int head_dim,
		      int page_size, const double *q_rot, const int32_t *block_tables,
		      int max_blocks, const int32_t *seq_lens, int batch, int num_q_heads,
		      double scale, double *out)
{
	if (num_kv_heads <= 0 || num_q_heads % num_kv_heads || head_dim <= 0)
		return -3;
	int g = num_q_heads / num_kv_heads;
	int nmax = max_blocks * page_size;
	double *kd = malloc(sizeof(double) * (size_t)nmax * head_dim);
	double *vd = malloc(sizeof(double) * (size_t)nmax * head_dim);
	double *s = malloc(sizeof(double) * (size_t)nmax);
	int rc = 0;
	if (!kd || !vd || !s) {
		rc = -4;
		goto done;
	}
	for (int b = 0; b < batch && !rc; b++) {
		int n = seq_lens[b];
		if (n < 1 || n > nmax) {
			rc = -1;
			break;
		}
		const int32_t *bt_row = block_tables + (size_t)b * max_blocks;
		for (int h = 0; h < num_kv_heads && !rc; h++) {
			rc = gather(pool, num_pages, num_kv_heads, head_dim, page_size, bt_row, h, 0, n,
				    kd, vd);
			for (int i = h * g; i < (h + 1) * g && !rc; i++) {
				size_t row = (size_t)b * num_q_heads + i;
				attend(q_rot + row * head_dim, kd, vd, n, head_dim, scale, s,
				       out + row * head_dim);
			}
		}
	}
done:
	free(kd);
	free(vd);
	free(s);
	return rc;
}

/* [P3] feature list: "prefill fills prompt pages" and the dense causal
 * prefill item; RoPE per [P2]. Chunked prefill of `batch` sequences: sequence
 * b holds start_pos[b] cached tokens and brings the chunk of tokens
 * cu_tokens[b] .. cu_tokens[b+1]-1 (rows of q, k, v, q_rot and out), at
 * positions start_pos[b], start_pos[b]+1, ... Every chunk token is rotated
 * and appended exactly as oracle_append_rope appends one decode token; then
 * the queries of chunk token t attend causally, over the first
 * start_pos[b] + t + 1 tokens of the sequence (the cached ones, the chunk's
 * earlier tokens and itself), exactly as oracle_gqa_decode attends for one
 * sequence of that length. */
int oracle_prefill(uint16_t *pool, long num_pages, int num_kv_heads, int head_dim,
		   int page_size, const uint16_t *q, const uint16_t *k, const uint16_t *v,
		   const int32_t *block_tables, int max_blocks, const int32_t *cu_tokens,
		   const int32_t *start_pos, int batch, int num_q_heads, double theta,
		   double scale, double *q_rot, double *out)
{
	int rc = 0;
	for (int pass = 0; pass < 2 && !rc; pass++) {
		for (int b = 0; b < batch && !rc; b++) {
			const int32_t *row = block_tables + (size_t)b * max_blocks;
			if (cu_tokens[b + 1] < cu_tokens[b] || start_pos[b] < 0)
				return -1;
			for (int idx = cu_tokens[b]; idx < cu_tokens[b + 1] && !rc; idx++) {
				int32_t pos = start_pos[b] + (idx - cu_tokens[b]);
				int32_t len = pos + 1;
				size_t qo = (size_t)idx * num_q_heads * head_dim;
				size_t ko = (size_t)idx * num_kv_heads * head_dim;
				if (pass == 0)
					rc = oracle_append_rope(pool, num_pages, num_kv_heads, head_dim,
								page_size, q + qo, k + ko, v + ko,
								q_rot + qo, row, max_blocks, &len, &pos, 1,
								num_q_heads, theta);
				else
					rc = oracle_gqa_decode(pool, num_pages, num_kv_heads, head_dim,
							       page_size, q_rot + qo, row, max_blocks,
							       &len, 1, num_q_heads, scale, out + qo);
			}
		}
	}
	return rc;
}

/*
 * Split-KV form (flash-decoding; not on the pages, defined by its closed
 * form): the tokens of each (b, i) row are cut into consecutive splits of
 * tokens_per_split; split j yields its own softmax-normalised output o_j and
 * the log-sum-exp of its scores lse_j. Row r = b*Hq + i has num_splits[r]
 * splits stored at o_part[(r*max_splits + j)*D], lse_part[r*max_splits + j].
 */
int oracle_gqa_decode_split(const uint16_t *pool, long num_pages, int num_kv_heads,
			    int head_dim, int page_size, const double *q_rot,
			    const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
			    int batch, int num_q_heads, double scale, int tokens_per_split,
			    int max_splits, double *o_part, double *lse_part, int32_t *num_splits)
{
	if (num_kv_heads <= 0 || num_q_heads % num_kv_heads || tokens_per_split <= 0)
		return -3;
	int g = num_q_heads / num_kv_heads;
	int nmax = max_blocks * page_size;
	double *kd = malloc(sizeof(double) * (size_t)nmax * head_dim);
	double *vd = malloc(sizeof(double) * (size_t)nmax * head_dim);
	double *s = malloc(sizeof(double) * (size_t)nmax);
	int rc = 0;
	if (!kd || !vd || !s) {
		rc = -4;
		goto done;
	}
	for (int b = 0; b < batch && !rc; b++) {
		int n = seq_lens[b];
		if (n < 1 || n > nmax) {
			rc = -1;
			break;
		}
		int nsplit = (n + tokens_per_split - 1) / tokens_per_split;
		if (nsplit > max_splits) {
			rc = -3;
			break;
		}
		const int32_t *bt_row = block_tables + (size_t)b * max_blocks;
		for (int h = 0; h < num_kv_heads && !rc; h++) {
			rc = gather(pool, num_pages, num_kv_heads, head_dim, page_size, bt_row, h, 0, n,
				    kd, vd);
			for (int i = h * g; i < (h + 1) * g && !rc; i++) {
				size_t row = (size_t)b * num_q_heads + i;
				num_splits[row] = nsplit;
				for (int j = 0; j < nsplit; j++) {
					int t0 = j * tokens_per_split;
					int t1 = t0 + tokens_per_split < n ? t0 + tokens_per_split : n;
					size_t slot = row * max_splits + j;
					lse_part[slot] = attend(q_rot + row * head_dim,
								kd + (size_t)t0 * head_dim,
								vd + (size_t)t0 * head_dim, t1 - t0,
								head_dim, scale, s,
								o_part + slot * head_dim);
				}
			}
		}
	}
done:
	free(kd);
	free(vd);
	free(s);
	return rc;
}

/* Log-sum-exp merge of split results (closed form): with M = max_j lse_j and
 * w_j = exp(lse_j - M), out = sum_j w_j o_j / sum_j w_j. */
void oracle_lse_combine(const double *o_part, const double *lse_part, const int32_t *num_splits,
			int rows, int max_splits, int head_dim, double *out)
{
	for (int r = 0; r < rows; r++) {
		int ns = num_splits[r];
		double m = -INFINITY;
		for (int j = 0; j < ns; j++)
			if (lse_part[(size_t)r * max_splits + j] > m)
				m = lse_part[(size_t)r * max_splits + j];
		double wsum = 0.0;
		for (int d = 0; d < head_dim; d++)
			out[(size_t)r * head_dim + d] = 0.0;
		for (int j = 0; j < ns; j++) {
			size_t slot = (size_t)r * max_splits + j;
			double w = exp(lse_part[slot] - m);
			wsum += w;
			for (int d = 0; d < head_dim; d++)
				out[(size_t)r * head_dim + d] += w * o_part[slot * head_dim + d];
		}
		for (int d = 0; d < head_dim; d++)
			out[(size_t)r * head_dim + d] /= wsum;
	}
}
