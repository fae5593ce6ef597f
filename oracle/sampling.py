"""Modified rejection sampling for a batch of ragged sequences, in float64.

TEST INFRASTRUCTURE ONLY: part of the CPU oracle.  Only tests, the smoke check
and the bench's CPU-baseline leg may import it.

Method source: "Accelerating Large Language Model Decoding with Speculative
Sampling" (Chen et al.; called SpS below):
  * section "Modified rejection sampling" (改进的拒绝采样): accept draft x~ with
    probability min(1, q(x~)/p(x~)); go left to right and stop at the first
    rejection; on rejection resample from (q - p)_+ = max(0, q-p)/sum max(0, q-p);
    if every draft is accepted, sample one more token from the last target row
    (at least one and at most K+1 tokens per loop);
  * same section, "compatibility with standard sampling methods": temperature /
    nucleus / top-k change the probabilities *before* the rejection scheme;
  * appendix "Proof", Theorem 1: the scheme recovers q exactly.
Batch shape (ragged draft counts, no padding): "EMS-SD: Efficient Multi-sample
Speculative Decoding" abstract; "BASS: Batched Attention-optimized Speculative
Sampling" abstract.

Readings where the pages are silent (each one is listed in the design notes):
  * the compare is `u * p_hat(x~) < q_hat(x~)` with u in [0,1): for p_hat > 0
    this is u < min(1, q/p) with no division, p == q always accepts, and for
    p_hat == 0 the draft is accepted iff q_hat > 0;
  * temperature first (z = logit / T), then top-k, then nucleus on the
    renormalized top-k distribution (the usual order of these transforms);
    top-k keeps {x : z_x >= tau_k}, tau_k the k-th largest value of z counted
    with multiplicity (ties at the boundary kept); the nucleus keeps
    {x : z_x >= tau}, tau the largest attained value whose upper set holds
    mass >= top_p (tie-inclusive, no index tie-break);
  * temperature 0 is greedy decoding: the processed row is one-hot at the
    first (lowest-index) maximum of the logits, and the accept / residual
    rules then keep a draft iff it is that argmax;
  * per-sequence temperature / top_p / top_k arrays override the scalars; an
    invalid per-sequence value (T < 0 or NaN, top_p <= 0 or NaN, top_k < 0)
    makes that sequence fail with the NONFINITE and BAD_PARAM bits;
  * the same processing is applied to q and p;
  * the inverse-CDF draw walks the vocabulary in index order and takes the first
    x whose cumulative weight exceeds u * Z (strict, so zero weights are never
    chosen); if a rejection leaves Z == 0 the draw falls back to q_hat and the
    EMPTY_RESIDUAL status bit is set;
  * a draft token outside [0, V) is a rejection with the BAD_TOKEN bit;
  * a row holding NaN or +inf, or only -inf, makes its sequence fail (no token,
    no append, NONFINITE bit) when the left-to-right loop reaches it: target
    and draft row j up to the first rejection, or the bonus row; rows after
    the first rejection are never used (the loop stops there), so they cannot
    fail the sequence.
"""
import numpy as np

from .philox import verify_uniforms

# Device-status bits (same meaning as the C-ABI's bits; values restated here).
DEV_CAPACITY = 1
DEV_BAD_TOKEN = 2
DEV_NONFINITE = 4
DEV_EMPTY_RESIDUAL = 8
DEV_BAD_LENGTH = 16
DEV_BAD_PARAM = 64

# Near-tie audit windows.  Decisions this close to a boundary may legitimately
# differ between an fp32 GPU path and this fp64 oracle; they are counted and
# excluded from bit-exact comparison (with everything after them in that
# sequence).  TIE_EPS is the stated window of the accept compare and of the
# residual / bonus CDF at the drawn token.
TIE_EPS = 1e-5
# Nucleus cut window: the cut compares a mass with top_p; an fp32 path (fp32
# weights, exact sums of them) gets that mass to ~5e-7, so boundaries within
# 2e-6 of top_p are treated as ties (the 1e-5 windows above are for u
# comparisons).
NUCLEUS_TIE_EPS = 2e-6
TIE_ACCEPT = 1
TIE_DRAW = 2


# --------------------------------------------------------------------------
# exact conversions of the stored inputs
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits):
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes):
    """8-bit E4M3 codes (uint8) -> float64, exactly.

    The format (the 8-bit floating point KV caches use; the OCP FP8 "E4M3"
    layout): sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
    0 holds the subnormals m/8 * 2^-6; no infinities, and S.1111.111 is NaN, so
    the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def to_f64(x):
    """Stored tensor (float32 array, uint16 bfloat16 bits or uint8 E4M3 codes)
    -> float64 exactly."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    if x.dtype == np.uint8:
        return e4m3_to_f64(x)
    return x.astype(np.float64)


# --------------------------------------------------------------------------
# probability processing (SpS, "compatibility with standard sampling methods")
# --------------------------------------------------------------------------
class ProcessedRow:
    """One processed logits row.

    probs:   float64 [V], the processed distribution (0 outside the nucleus)
    valid:   False if the row held NaN/+inf or only -inf
    tau:     nucleus threshold on z (-inf when top_p >= 1)
    margin:  distance of the nucleus boundary masses from top_p (inf if none)
    """
    __slots__ = ("probs", "valid", "tau", "margin")

    def __init__(self, probs, valid, tau, margin):
        self.probs, self.valid, self.tau, self.margin = probs, valid, tau, margin


def params_ok(temperature, top_p, top_k):
    """Valid processing parameters (as float32 / int32 values)."""
    T = float(np.float32(temperature))
    tp = float(np.float32(top_p))
    return T >= 0.0 and tp > 0.0 and int(top_k) >= 0


def process_row(logits, temperature, top_p, top_k=0, alt=False):
    """Temperature, then top-k, then nucleus, on one row of exact float64
    logits; temperature 0 is greedy (one-hot at the first maximum).

    temperature and top_p are taken as the float32 values the C-ABI receives.
    With alt=True, a row whose nucleus boundary mass lies within
    NUCLEUS_TIE_EPS of top_p is returned with the neighbouring cut instead
    (one tie class more when the kept mass barely reaches top_p, one fewer
    when the mass above the cut barely misses it): the row a path whose mass
    sums differ by rounding may build.  Other rows are returned unchanged.
    """
    T = float(np.float32(temperature))
    tp = float(np.float32(top_p))
    k = int(top_k)
    l = np.asarray(logits, dtype=np.float64)
    V = l.shape[0]
    if np.any(np.isnan(l)) or np.any(l == np.inf) or not np.any(l > -np.inf):
        return ProcessedRow(np.zeros(V), False, np.nan, np.inf)
    if T == 0.0:                         # greedy
        probs = np.zeros(V)
        x = int(np.argmax(l))            # first maximum
        probs[x] = 1.0
        return ProcessedRow(probs, True, l[x], np.inf)
    z = l / T
    w = np.exp(z - z.max())              # exp(-inf) = 0 for masked entries
    tau_k = -np.inf
    if 0 < k < V:
        tau_k = np.sort(z)[::-1][k - 1]  # k-th largest, with multiplicity
        w = np.where(z >= tau_k, w, 0.0)
    if tp >= 1.0:
        return ProcessedRow(w / w.sum(), True, tau_k, np.inf)
    P = w / w.sum()
    # Tie classes of equal z, highest first; upper-set masses M_k.
    vals, inv = np.unique(z, return_inverse=True)
    cls_mass = np.bincount(inv.ravel(), weights=P, minlength=vals.shape[0])
    vals, cls_mass = vals[::-1], cls_mass[::-1]
    M = np.cumsum(cls_mass)
    k = int(np.argmax(M >= tp)) if np.any(M >= tp) else vals.shape[0] - 1
    tau = vals[k]
    above = M[k] - tp
    # the mass above the top class is exactly 0 on every path: no tie there
    below = tp - M[k - 1] if k > 0 else np.inf
    if alt and min(abs(above), abs(below)) < NUCLEUS_TIE_EPS:
        if abs(above) <= abs(below) and k + 1 < vals.shape[0]:
            tau = vals[k + 1]
        elif k > 0:
            tau = vals[k - 1]
    keep = z >= tau
    wk = np.where(keep, w, 0.0)
    return ProcessedRow(wk / wk.sum(), True, tau, min(abs(above), abs(below)))


# --------------------------------------------------------------------------
# the three primitive decisions (SpS, "Modified rejection sampling")
# --------------------------------------------------------------------------
def accept(u_acc, p_of_draft, q_of_draft):
    """Accept the draft iff u * p(x~) < q(x~), i.e. with prob. min(1, q/p)."""
    return u_acc * p_of_draft < q_of_draft


def residual(q_row, p_row):
    """Unnormalized residual max(0, q - p) over the vocabulary."""
    return np.maximum(0, q_row - p_row)


def sample_index(weights, u):
    """Inverse CDF in index order: first x with sum_{y<=x} w_y > u * Z.

    Works on float64 arrays and on object arrays of Fractions; `u` may be an
    array (vectorized draw).  Returns None when Z <= 0.
    """
    c = np.cumsum(weights)               # sequential, left to right
    Z = c[-1]
    if not Z > 0:
        return None
    idx = np.searchsorted(c, u * Z, side="right")
    return idx if np.ndim(idx) else int(idx)


def _cdf_margin(weights, x, u):
    """Distance of u from the two ends of x's normalized CDF interval, Z, and
    the weighted tokens whose normalized CDF interval meets [u - TIE_EPS,
    u + TIE_EPS] (the draws a path whose CDF is off by less than TIE_EPS can
    make; x among them)."""
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    Z = c[-1]
    hi = c[x] / Z
    lo = c[x - 1] / Z if x > 0 else 0.0
    cn = c / Z
    lo_all = np.concatenate([[0.0], cn[:-1]])
    near = (w > 0) & (cn > u - TIE_EPS) & (lo_all <= u + TIE_EPS)
    return min(u - lo, hi - u), Z, {int(t) for t in np.flatnonzero(near)} | {int(x)}


# --------------------------------------------------------------------------
# one sequence
# --------------------------------------------------------------------------
def verify_sequence(q_rows, p_rows, drafts, u_acc, u_smp, audit=None):
    """Left-to-right accept loop, then residual or bonus draw.

    q_rows: [K+1, V] processed target rows; p_rows: [K, V] processed draft rows;
    drafts: [K] tokens; u_acc, u_smp: [K+1] uniforms for rows 0..K.
    Returns (n_accepted, sampled_token, status_bits).  If `audit` is a list, one
    (row, kind, margin, window) tuple is appended per decision taken; kind
    is "accept", "residual", "bonus" or "empty" (a rejection whose residual is
    zero everywhere: the draw then takes q_hat), window (draws only) the
    weighted tokens whose normalized CDF interval lies within TIE_EPS of u.
    """
    K = len(drafts)
    V = q_rows.shape[1] if hasattr(q_rows, "shape") else len(q_rows[0])
    status = 0
    for j in range(K):
        d = int(drafts[j])
        if d < 0 or d >= V:
            status |= DEV_BAD_TOKEN
            if audit is not None:
                audit.append((j, "accept", np.inf, None))
            break
        pd, qd = p_rows[j][d], q_rows[j][d]
        ok = accept(u_acc[j], pd, qd)
        if audit is not None:
            if pd > 0:
                ratio = min(1.0, float(qd) / float(pd))
                audit.append((j, "accept", abs(float(u_acc[j]) - ratio), None))
            else:
                audit.append((j, "accept", np.inf, None))
        if not ok:
            break
    else:
        j = K
    n = j
    kind = "bonus"
    if n < K:
        kind = "residual"
        w = residual(q_rows[n], p_rows[n])
        x = sample_index(w, u_smp[n])
        if x is None:                      # rejected, yet no positive residual
            status |= DEV_EMPTY_RESIDUAL
            kind = "empty"
            w = q_rows[n]
            x = sample_index(w, u_smp[n])
    else:
        w = q_rows[K]
        x = sample_index(w, u_smp[K])
    if audit is not None:
        m, Z, nb = _cdf_margin(w, x, float(u_smp[n]))
        audit.append((n, kind, m, nb))
    return n, x, status


def _first_rejection(qp, pp, drafts, u_acc, upto):
    """Index of the first rejected draft among pairs 0..upto-1 (all valid), or
    None when every one of them is accepted."""
    V = qp[0].probs.shape[0]
    for j in range(upto):
        d = int(drafts[j])
        if d < 0 or d >= V or not accept(u_acc[j], pp[j].probs[d], qp[j].probs[d]):
            return j
    return None


# --------------------------------------------------------------------------
# the batch
# --------------------------------------------------------------------------
def reject_sample(target_logits, draft_logits, draft_tokens, cu_q, kv_len,
                  temperature, top_p, seed, seq_ids=None, top_k=0, temperatures=None,
                  top_ps=None, top_ks=None):
    """Batched verify sampling over ragged sequences (no padding).

    target_logits [R, V], draft_logits [R-B, V] (stored float32 or bf16 bits);
    rows of sequence i: target cu_q[i] + j (j = 0..K_i), draft cu_q[i] - i + j
    (j = 0..K_i-1); draft_tokens [R-B] indexed like the draft rows.
    Row j decides token index pos = kv_len[i] + j + 1 with Philox uniforms
    keyed by (seed, seq_id, pos).  temperatures / top_ps / top_ks ([B] or
    None) override temperature / top_p / top_k per sequence.

    Returns dict with num_accepted [B] (-1 for a failed sequence), out_tokens
    [R] (drafts for j < n_i, the sampled token at j = n_i, -1 after; all -1 for
    a failed sequence), status (OR of bits), seq_status [B], and the near-tie
    audit:
      tie_row [B]   row of the first decision inside a tie window, or -1;
      tie_kind [B]  0 none, TIE_ACCEPT (an accept/reject decision, or a row
                    whose nucleus cut is itself a tie: rows before tie_row are
                    still exact), TIE_DRAW (the final draw: n_i, the accepted
                    drafts and the append are still exact);
      tie_alts      {i: set of tokens a draw tie may yield} for every TIE_DRAW
                    sequence: the weighted tokens whose normalized CDF interval
                    lies within TIE_EPS of u (the oracle's token among them);
      tie_count     number of sequences with a tie;
      tie_clauses   {"accept", "cdf", "nucleus"}: sequences whose first tie is
                    of that clause;
      tie_positions decisions inside a tie window along the oracle's own path
                    (a sequence can hold more than one).
    A decision is inside a tie window when |u - min(1, q/p)| < TIE_EPS, when
    the draw's normalized CDF interval has an end within TIE_EPS of u, or when
    a row it uses has a nucleus boundary mass within NUCLEUS_TIE_EPS of top_p.
    """
    cu_q = np.asarray(cu_q, dtype=np.int64)
    B = cu_q.shape[0] - 1
    R = int(cu_q[-1])
    kv_len = np.asarray(kv_len, dtype=np.int64)
    if seq_ids is None:
        seq_ids = np.arange(B, dtype=np.int64)
    num_acc = np.zeros(B, dtype=np.int32)
    out_tokens = np.full(R, -1, dtype=np.int32)
    seq_status = np.zeros(B, dtype=np.uint32)
    tie_row = np.full(B, -1, dtype=np.int64)
    tie_kind = np.zeros(B, dtype=np.int64)
    tie_alts = {}
    tie_count = 0
    tie_clauses = {"accept": 0, "cdf": 0, "nucleus": 0}
    tie_positions = 0
    for i in range(B):
        r0, r1 = int(cu_q[i]), int(cu_q[i + 1])
        K = r1 - r0 - 1
        p0 = r0 - i
        pos = kv_len[i] + np.arange(K + 1, dtype=np.int64) + 1
        u_acc, u_smp = verify_uniforms(seed, seq_ids[i], pos)
        T_i = temperature if temperatures is None else temperatures[i]
        tp_i = top_p if top_ps is None else top_ps[i]
        tk_i = top_k if top_ks is None else top_ks[i]
        if not params_ok(T_i, tp_i, tk_i):
            seq_status[i] = DEV_NONFINITE | DEV_BAD_PARAM
            num_acc[i] = -1
            continue
        qp = [process_row(to_f64(target_logits[r0 + j]), T_i, tp_i, tk_i)
              for j in range(K + 1)]
        pp = [process_row(to_f64(draft_logits[p0 + j]), T_i, tp_i, tk_i)
              for j in range(K)]
        # Only the row pairs the left-to-right loop reaches are used: pair j
        # (target row j, draft row j) up to the first rejection, or the bonus
        # row K.  The sequence fails if a reached row is invalid.
        bad_at = next((j for j in range(K + 1)
                       if not qp[j].valid or (j < K and not pp[j].valid)), None)
        Kr = K
        if bad_at is not None:
            rej = _first_rejection(qp, pp, draft_tokens[p0:p0 + K], u_acc, bad_at)
            if rej is None:                  # the loop reaches the invalid pair
                seq_status[i] = DEV_NONFINITE
                num_acc[i] = -1
                continue
            Kr = rej + 1                     # decisions 0..rej; rejected at rej
        audit = []
        V = qp[0].probs.shape[0]
        n, x, st = verify_sequence(np.stack([r.probs for r in qp[:Kr + 1]]),
                                   np.stack([r.probs for r in pp[:Kr]]) if Kr else
                                   np.zeros((0, V)),
                                   draft_tokens[p0:p0 + Kr], u_acc[:Kr + 1], u_smp[:Kr + 1],
                                   audit)
        seq_status[i] = st
        num_acc[i] = n
        out_tokens[r0:r0 + n] = draft_tokens[p0:p0 + n]
        out_tokens[r0 + n] = x
        # decisions inside a tie window (including nucleus boundaries of the
        # rows each decision used); the first one decides what stays exact
        first = True
        for (j, kind, m, nb) in audit:
            nuc = qp[j].margin if kind == "bonus" else min(
                qp[j].margin, pp[j].margin if j < K else np.inf)
            if not (m < TIE_EPS or nuc < NUCLEUS_TIE_EPS):
                continue
            tie_positions += 1
            if not first:
                continue
            first = False
            tie_row[i] = j
            tie_count += 1
            if nuc < NUCLEUS_TIE_EPS:
                tie_kind[i] = TIE_ACCEPT
                tie_clauses["nucleus"] += 1
            elif kind == "accept":
                tie_kind[i] = TIE_ACCEPT
                tie_clauses["accept"] += 1
            else:
                tie_kind[i] = TIE_DRAW
                tie_clauses["cdf"] += 1
                tie_alts[i] = set(nb)
    status = int(np.bitwise_or.reduce(seq_status)) if B else 0
    return dict(num_accepted=num_acc, out_tokens=out_tokens, status=status,
                seq_status=seq_status, tie_row=tie_row, tie_kind=tie_kind,
                tie_alts=tie_alts, tie_count=tie_count, tie_clauses=tie_clauses,
                tie_positions=tie_positions)
