"""Plain float64 CPU oracle for TurboQuant (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import this module.  It shares no code, constant table or
helper with the CUDA library; the library re-derives everything on its own.

Source: "Вечная математика TurboQuant: как сжать KV-кэш до предела Шеннона"
(blog.sergeynikolenko.ru, post 11266).  Section names below are that page's.

Parity pins (tests/test_oracle_pins.py) and status per function
---------------------------------------------------------------
splitmix64 / gaussian_matrix   pinned: SplitMix64 known-answer outputs for seed 0;
                               Box-Muller sample moments and a KS test vs N(0,1).
rotation_matrix (Π)            pinned: orthogonality to 1e-12; sign convention
                               diag(R) > 0 checked against a re-factorisation.
hadamard_matrix /              pinned: H equals scipy.linalg.hadamard; Π x equals an
hadamard_rotation (Π_H)        in-place butterfly transform of σ∘x over √d; one-hot
                               rows give the closed-form b = 1 distortion
                               (1 − √d·c₁)²; Gaussian rows keep D_mse = d·C(f_X,b).
coord_density / cdf / moment   pinned: density integrates to 1 (quadrature), the
                               b=1 centroid equals the closed form
                               Γ(d/2)/(√π Γ((d+1)/2)), Gaussian limit at large d.
lloyd_max_codebook             pinned: fixed-point residual vs independent
                               quadrature, page values ±0.453/√d, ±1.51/√d, the
                               Gaussian Lloyd–Max table of Max (1960) at large d.
quantize / dequantize (mse)    pinned: empirical D_mse equals d·C(f_X,b) (exact
                               identity of the Theorem 1 proof sketch), the page's
                               D_mse table, Shannon and Panter–Dite bounds, b=1 bias
                               factor d·c₁² (→2/π), brute-force nearest codeword at
                               d=4/8.
quantize / dequantize (prod)   pinned: unbiasedness over seeds, exact b=1 variance
                               ((π/2)‖y‖² − ⟨x,y⟩²)/d, D_prod ≤ (π/2)·D_mse(b−1).
pack_codes / pack_signs        pinned: hand-written golden bytes
                               (tests/golden/pack_layout.txt), round trip.
mixed_* (outlier channels)     pinned: the page's split counts (32·3 + 96·2)/128 =
                               2.25 code bits per channel; distortion = ‖x_O‖²·D_mse(d_o, b_o) +
                               ‖x_N‖²·D_mse(d_n, b_n) on Gaussian rows; channel
                               relabelling equivariance; scores are the sums of the
                               two parts' scores from decode_attention; planted
                               outlier channels are the ones selected.
decode_attention               pinned: q = 0 gives the plain mean of dequantized
                               values, one-token context returns that value,
                               brute-force loop on a tiny case, dequant-free
                               rotated-domain identity of the score.

Readings where the page is silent
---------------------------------
* "Gaussian" means i.i.d. N(0,1) entries (Шаг 1, QJL).  Π and S come from two
  independent streams (community finding #3 on the page).
* Random numbers: SplitMix64 (counter form: output i mixes seed + (i+1)·φ64),
  uniform u = (z >> 11)·2⁻⁵³, Box–Muller on consecutive pairs (u₁ = 0 → 2⁻⁵³),
  matrices filled row-major.  Stream seeds: seed ⊕ PI_STREAM_TAG for Π,
  seed ⊕ S_STREAM_TAG for S.
* Π = Q·diag(sign(R_ii)) from G = QR (makes Π Haar-distributed).
* Walsh–Hadamard option (community finding #3 names WHT for the MSE stage and an
  independent transform for QJL, without defining the randomisation): the
  standard randomised Hadamard transform Π_H = H_d·diag(σ)/√d, H_d the Sylvester
  (natural-order) Hadamard matrix, σ_i = +1 if u_i < ½ else −1 with u_i the i-th
  uniform of stream seed ⊕ WHT_STREAM_TAG.  d must be a power of two.  S stays
  Gaussian from its own stream.
* Codebook uses the exact coordinate law f_X, not its N(0, 1/d) limit.
* Ties y_j = t_k go to the lower index; sign(0) = +1; a zero row stores norm 0,
  codes 0, signs +1, residual norm 0 (dequantizes to 0).
* Norms are stored as float32 ("as a float", Шаг 0); dequantization uses the
  stored float32 values.
* prod with b = 1 has a 0-bit MSE stage: one level at 0, residual r = x̂.
* Attention: contiguous GQA (query head h reads KV head h // (Hq/Hkv)),
  scale 1/√d by default, no causal mask, empty context → output 0.
* Outlier channels (experiments section, 32 channels at 3 bits + 96 at 2; the
  page's sum (32·3 + 96·2)/128 is 2.25, not the 2.5 it prints — 2.5 counts two
  16-bit part norms as well; the split is kept as printed): each
  part of a row gets its own TurboQuant quantizer (own norm, rotation, codebook);
  the page does not say how the outlier channels are found, so they are the d_o
  channels of largest energy over the rows being cached.
"""
from __future__ import annotations

import math

import numpy as np
from scipy import special

__all__ = [
    "PI_STREAM_TAG", "S_STREAM_TAG", "splitmix64", "uniform01", "gaussian_matrix",
    "WHT_STREAM_TAG", "ROTATIONS", "rotation_matrix", "hadamard_matrix", "hadamard_signs",
    "hadamard_rotation", "qjl_matrix", "coord_density_const", "coord_density",
    "coord_cdf", "cell_mass", "cell_first_moment", "lloyd_max_codebook",
    "mse_distortion_theory", "Params", "make_params", "quantize", "qjl_of_residual", "pack_codes",
    "unpack_codes", "pack_signs", "unpack_signs", "dequantize", "decode_attention",
    "code_bytes_per_row", "sign_bytes_per_row", "MixedParams", "outlier_channel_perm",
    "mixed_bits_per_channel", "mixed_quantize", "mixed_dequantize", "mixed_decode_attention",
]

MASK64 = (1 << 64) - 1
GOLDEN64 = 0x9E3779B97F4A7C15
# Independent streams for the rotation and the QJL matrix (arbitrary distinct tags).
PI_STREAM_TAG = 0x5049524F54415445  # "PIROTATE"
S_STREAM_TAG = 0x514A4C534B455443  # "QJLSKETC"
WHT_STREAM_TAG = 0x5748545349474E53  # "WHTSIGNS": the ±1 diagonal of the Hadamard rotation
ROTATIONS = ("qr", "hadamard")


# ----------------------------------------------------------------------------
# Random numbers (page silent: build-defined, published SplitMix64 + Box-Muller)
# ----------------------------------------------------------------------------
def splitmix64(seed: int, count: int) -> np.ndarray:
    """First ``count`` SplitMix64 outputs for ``seed`` (Steele, Lea & Flood 2014).

    Counter form: state_i = seed + (i+1)·0x9E3779B97F4A7C15 (mod 2^64), then the
    published 64-bit finaliser.
    """
    i = np.arange(1, count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + i * np.uint64(GOLDEN64)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, count: int) -> np.ndarray:
    """u = (z >> 11)·2⁻⁵³ in [0, 1)."""
    z = splitmix64(seed, count)
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def gaussian_matrix(seed: int, rows: int, cols: int) -> np.ndarray:
    """i.i.d. N(0,1) matrix, row-major, Box–Muller on consecutive uniform pairs."""
    n = rows * cols
    npairs = (n + 1) // 2
    u = uniform01(seed, 2 * npairs)
    u1 = u[0::2].copy()
    u2 = u[1::2]
    u1[u1 == 0.0] = 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    g = np.empty(2 * npairs)
    g[0::2] = r * np.cos(2.0 * math.pi * u2)
    g[1::2] = r * np.sin(2.0 * math.pi * u2)
    return g[:n].reshape(rows, cols)


# ----------------------------------------------------------------------------
# Шаг 1: random rotation Π = orthogonal factor of a Gaussian matrix
# ----------------------------------------------------------------------------
def rotation_matrix(d: int, seed: int) -> np.ndarray:
    """Π ∈ R^{d×d} from the QR decomposition of a Gaussian matrix (Шаг 1).

    Sign convention (page silent): Π = Q·diag(sign(R_ii)), which makes the factor
    unique and Haar distributed.
    """
    G = gaussian_matrix(seed ^ PI_STREAM_TAG, d, d)
    Q, R = np.linalg.qr(G)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s[None, :]


def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d (natural order): H_1 = [1], H_2m = [[H, H], [H, −H]]."""
    assert d >= 1 and d & (d - 1) == 0, "d must be a power of two"
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def hadamard_signs(d: int, seed: int) -> np.ndarray:
    """Random ±1 diagonal σ of the Hadamard rotation: σ_i = +1 iff u_i < ½."""
    u = uniform01(seed ^ WHT_STREAM_TAG, d)
    return np.where(u < 0.5, 1.0, -1.0)


def hadamard_rotation(d: int, seed: int) -> np.ndarray:
    """Randomised Walsh–Hadamard rotation Π_H = H_d·diag(σ)/√d (orthogonal)."""
    return hadamard_matrix(d) * hadamard_signs(d, seed)[None, :] / math.sqrt(d)


def qjl_matrix(d: int, seed: int) -> np.ndarray:
    """S ∈ R^{d×d} with i.i.d. N(0,1) entries (section «QJL»)."""
    return gaussian_matrix(seed ^ S_STREAM_TAG, d, d)


# ----------------------------------------------------------------------------
# Lemma: coordinate law on the sphere, f_X(x) = Γ(d/2)/(√π Γ((d−1)/2)) (1−x²)^((d−3)/2)
# ----------------------------------------------------------------------------
def coord_density_const(d: int) -> float:
    return math.exp(math.lgamma(d / 2.0) - 0.5 * math.log(math.pi) - math.lgamma((d - 1) / 2.0))


def coord_density(x, d: int):
    x = np.asarray(x, dtype=np.float64)
    return coord_density_const(d) * np.power(np.clip(1.0 - x * x, 0.0, None), (d - 3) / 2.0)


def coord_cdf(x, d: int):
    """F(x) = I_{(x+1)/2}((d−1)/2, (d−1)/2): with u = (x+1)/2, f_X dx is Beta((d−1)/2, (d−1)/2)."""
    a = (d - 1) / 2.0
    u = (np.asarray(x, dtype=np.float64) + 1.0) / 2.0
    return special.betainc(a, a, np.clip(u, 0.0, 1.0))


def cell_mass(lo: float, hi: float, d: int) -> float:
    """∫_lo^hi f_X, using the symmetry F(−x) = 1 − F(x) on the upper side to avoid cancellation."""
    if lo >= 0.0:
        return float(coord_cdf(-lo, d) - coord_cdf(-hi, d))
    return float(coord_cdf(hi, d) - coord_cdf(lo, d))


def cell_first_moment(lo: float, hi: float, d: int) -> float:
    """∫_lo^hi x f_X(x) dx = C_d/(d−1)·[(1−lo²)^((d−1)/2) − (1−hi²)^((d−1)/2)] (antiderivative)."""
    c = coord_density_const(d) / (d - 1)
    p = (d - 1) / 2.0
    return c * (max(1.0 - lo * lo, 0.0) ** p - max(1.0 - hi * hi, 0.0) ** p)


# ----------------------------------------------------------------------------
# Шаг 2: Lloyd–Max scalar quantizer C(f_X, b)
# ----------------------------------------------------------------------------
def lloyd_max_codebook(d: int, levels: int, tol: float | None = None, max_iter: int = 100000):
    """1-D continuous k-means on [−1, 1] for f_X with ``levels`` cells (Шаг 2).

    Alternates the two optimality conditions the page states: boundaries are the
    midpoints of neighbouring centroids, centroids are the conditional means of
    f_X on their cells.  Starts from the N(0, 1/d) quantiles and stops when the
    centroids no longer move (the fixed point is unique: f_X is log-concave).

    Returns (centroids [levels], boundaries [levels−1]).
    """
    if levels == 1:
        return np.zeros(1), np.zeros(0)
    sigma = 1.0 / math.sqrt(d)
    if tol is None:
        # float64 noise floor of one update is ~1e-15 at the d = 128 scale
        tol = 3e-15 * max(1.0, math.sqrt(128.0 / d))
    c = sigma * special.ndtri((np.arange(levels) + 0.5) / levels)
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-1.0], t, [1.0]))
        c_new = np.array([cell_first_moment(edges[i], edges[i + 1], d) / cell_mass(edges[i], edges[i + 1], d)
                          for i in range(levels)])
        delta = np.max(np.abs(c_new - c))
        c = c_new
        if delta <= tol:
            break
    t = 0.5 * (c[:-1] + c[1:])
    return c, t


def mse_distortion_theory(d: int, levels: int) -> float:
    """D_mse = d·C(f_X, b) (Theorem 1 proof sketch).  With centroids at the
    conditional means, C = E[X²] − Σ_i c_i² P_i and E[X²] = 1/d."""
    c, t = lloyd_max_codebook(d, levels)
    edges = np.concatenate(([-1.0], t, [1.0]))
    mass = np.array([cell_mass(edges[i], edges[i + 1], d) for i in range(levels)])
    return 1.0 - d * float(np.sum(c * c * mass))


# ----------------------------------------------------------------------------
# Parameters of one quantizer (one handle)
# ----------------------------------------------------------------------------
class Params:
    """Everything a TurboQuant quantizer is determined by: (d, b, variant, seed)."""

    def __init__(self, d, bits, variant, seed, Pi, S, centroids, bounds, rotation="qr"):
        self.d = d
        self.rotation = rotation  # "qr" (Шаг 1) or "hadamard"
        self.bits = bits
        self.variant = variant  # "mse" or "prod"
        self.seed = seed
        self.Pi = Pi
        self.S = S
        self.centroids = centroids
        self.bounds = bounds
        self.b_mse = bits if variant == "mse" else bits - 1
        self.levels = 1 << self.b_mse
        self.gamma = math.sqrt(math.pi / 2.0) / d  # QJL dequantizer scale √(π/2)/d


_CODEBOOK_CACHE: dict = {}


def make_params(d: int, bits: int, variant: str, seed: int, rotation: str = "qr") -> Params:
    assert variant in ("mse", "prod") and rotation in ROTATIONS
    b_mse = bits if variant == "mse" else bits - 1
    key = (d, 1 << b_mse)
    if key not in _CODEBOOK_CACHE:
        _CODEBOOK_CACHE[key] = lloyd_max_codebook(d, 1 << b_mse)
    c, t = _CODEBOOK_CACHE[key]
    Pi = rotation_matrix(d, seed) if rotation == "qr" else hadamard_rotation(d, seed)
    S = qjl_matrix(d, seed) if variant == "prod" else None
    return Params(d, bits, variant, seed, Pi, S, c.copy(), t.copy(), rotation)


def code_bytes_per_row(p: Params) -> int:
    return p.b_mse * p.d // 8


def sign_bytes_per_row(p: Params) -> int:
    return p.d // 8 if p.variant == "prod" else 0


# ----------------------------------------------------------------------------
# Quantization: Шаг 0 (norm), Шаг 1 (rotate), Шаг 2 (nearest centroid),
# «Собственно TurboQuant» (QJL of the residual)
# ----------------------------------------------------------------------------
def quantize(p: Params, X) -> dict:
    """Quantize rows of X [n, d].

    Returns a dict with
      idx    [n, d] int   centroid index per rotated coordinate
      norm   [n] float32  ‖x‖ (Шаг 0)
      z      [n, d] ±1    QJL signs sign(S r) (prod only)
      rnorm  [n] float32  ‖r‖ of the unit-scale residual (prod only)
      y_unit [n, d]       rotated unit coordinates Πx̂ (for boundary margins)
      sr     [n, d]       S r before the sign (for sign margins; prod only)
    """
    X = np.asarray(X, dtype=np.float64)
    n_rows, d = X.shape
    assert d == p.d
    norm = np.sqrt(np.sum(X * X, axis=1))
    nz = norm > 0
    xhat = np.zeros_like(X)
    xhat[nz] = X[nz] / norm[nz, None]
    y = xhat @ p.Pi.T                                    # y = Π x̂
    idx = np.searchsorted(p.bounds, y, side="left")      # #{k : t_k < y_j}
    idx[~nz] = 0
    out = {"idx": idx.astype(np.int64), "norm": norm.astype(np.float32), "y_unit": y}
    if p.variant == "prod":
        out.update(qjl_of_residual(p, X, out["idx"]))
    return out


def qjl_of_residual(p: Params, X, idx) -> dict:
    """«Собственно TurboQuant» steps 2–3 for given mse indices: residual
    r = x̂ − Q_mse⁻¹(idx) = x̂ − Πᵀc[idx], then store sign(S·r) and ‖r‖."""
    X = np.asarray(X, dtype=np.float64)
    norm = np.sqrt(np.sum(X * X, axis=1))
    nz = norm > 0
    xhat = np.zeros_like(X)
    xhat[nz] = X[nz] / norm[nz, None]
    x_mse = p.centroids[np.asarray(idx)] @ p.Pi          # Q_mse⁻¹: rows of (Πᵀ c[idx])ᵀ
    r = xhat - x_mse                                     # residual r = x − Q_mse⁻¹(Q_mse(x))
    r[~nz] = 0.0
    sr = r @ p.S.T                                       # S r
    z = np.where(sr >= 0.0, 1, -1).astype(np.int8)       # sign, with sign(0) = +1
    return {"z": z, "rnorm": np.sqrt(np.sum(r * r, axis=1)).astype(np.float32), "sr": sr}


def pack_codes(idx, b_mse: int) -> np.ndarray:
    """Bit-pack per-coordinate indices, row by row: code j occupies bits
    [j·b, (j+1)·b) of the row, least significant bit first; bit k of the row is
    bit (k mod 8) of byte k div 8."""
    idx = np.asarray(idx, dtype=np.int64)
    n_rows, d = idx.shape
    if b_mse == 0:
        return np.zeros((n_rows, 0), dtype=np.uint8)
    bits = np.zeros((n_rows, d * b_mse), dtype=np.uint8)
    for pbit in range(b_mse):
        bits[:, pbit::b_mse] = (idx >> pbit) & 1
    return np.packbits(bits, axis=1, bitorder="little")


def unpack_codes(packed, d: int, b_mse: int) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    if b_mse == 0:
        return np.zeros((packed.shape[0], d), dtype=np.int64)
    bits = np.unpackbits(packed, axis=1, bitorder="little")[:, : d * b_mse].astype(np.int64)
    idx = np.zeros((packed.shape[0], d), dtype=np.int64)
    for pbit in range(b_mse):
        idx |= bits[:, pbit::b_mse] << pbit
    return idx


def pack_signs(z) -> np.ndarray:
    """Bit i of the row (LSB-first, as for codes) is 1 when z_i = +1."""
    z = np.asarray(z)
    return np.packbits((z > 0).astype(np.uint8), axis=1, bitorder="little")


def unpack_signs(packed, d: int) -> np.ndarray:
    bits = np.unpackbits(np.asarray(packed, dtype=np.uint8), axis=1, bitorder="little")[:, :d]
    return np.where(bits == 1, 1.0, -1.0)


def dequantize(p: Params, idx, norm, z=None, rnorm=None) -> np.ndarray:
    """x̃ = ‖x‖·(Πᵀ c[idx] + γ‖r‖ Sᵀ z): centroids rotated back by Πᵀ, plus for
    prod the QJL reconstruction √(π/2)/d·Sᵀz of the residual scaled by ‖r‖.
    Uses the stored float32 norms."""
    idx = np.asarray(idx, dtype=np.int64)
    x = p.centroids[idx] @ p.Pi                          # rows of (Πᵀ c[idx])ᵀ
    if p.variant == "prod":
        zf = np.asarray(z, dtype=np.float64)
        x = x + p.gamma * np.asarray(rnorm, dtype=np.float64)[:, None] * (zf @ p.S)
    return np.asarray(norm, dtype=np.float64)[:, None] * x


# ----------------------------------------------------------------------------
# Decode attention over the compressed cache (the page: prod needs a custom
# attention kernel; the math is plain softmax attention on dequantized K, V)
# ----------------------------------------------------------------------------
def decode_attention(pk: Params, pv: Params, q, k_rows: dict, v_rows: dict, seq_lens,
                     Hkv: int, T_max: int, scale: float | None = None):
    """Plain softmax attention of one decode query per head over dequantized keys
    and values.

    q        [B, Hq, d]
    k_rows   dict(idx, norm[, z, rnorm]) with rows ordered [B][Hkv][T_max]
    v_rows   same for values
    Returns (out [B, Hq, d] float64, scores [B, Hq, T_max] float64, NaN past seq_len).
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    K = dequantize(pk, k_rows["idx"], k_rows["norm"], k_rows.get("z"), k_rows.get("rnorm"))
    V = dequantize(pv, v_rows["idx"], v_rows["norm"], v_rows.get("z"), v_rows.get("rnorm"))
    K = K.reshape(B, Hkv, T_max, d)
    V = V.reshape(B, Hkv, T_max, d)
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, T_max), np.nan)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            kv = h // G
            if L == 0:
                continue
            s = scale * (K[b, kv, :L] @ q[b, h])
            scores[b, h, :L] = s
            w = np.exp(s - np.max(s))
            w /= np.sum(w)
            out[b, h] = w @ V[b, kv, :L]
    return out, scores


# ----------------------------------------------------------------------------
# Outlier-channel mixed precision (the page's experiments, KV cache: 32 outlier
# channels at 3 bits and the other 96 at 2 bits, (32·3 + 96·2)/128 = 2.25 code
# bits per channel; the page prints 2.5, which needs two 16-bit part norms)
# ----------------------------------------------------------------------------
class MixedParams:
    """Two independent quantizers over a split of the channels: ``po`` for the
    outlier channels ``perm[:po.d]`` and ``pn`` for the others ``perm[po.d:]``."""

    def __init__(self, po: Params, pn: Params, perm):
        perm = np.asarray(perm, dtype=np.int64)
        assert po.variant == pn.variant
        assert perm.shape == (po.d + pn.d,) and np.array_equal(np.sort(perm), np.arange(perm.size))
        self.po, self.pn, self.perm = po, pn, perm
        self.d = perm.size
        self.out = perm[: po.d]
        self.rest = perm[po.d:]


def outlier_channel_perm(X, d_o: int) -> np.ndarray:
    """Channel split (the page does not say how outliers are chosen): the d_o
    channels of largest energy Σ_rows x² (ties to the lower index), ascending,
    then the other channels ascending."""
    X = np.asarray(X, dtype=np.float64)
    e = np.sum(X * X, axis=0)
    order = sorted(range(X.shape[1]), key=lambda j: (-e[j], j))
    out = np.sort(np.asarray(order[:d_o], dtype=np.int64))
    rest = np.setdiff1d(np.arange(X.shape[1]), out)
    return np.concatenate([out, rest])


def mixed_bits_per_channel(mp: MixedParams) -> float:
    """(d_o·b_o + d_n·b_n)/d: code bits per channel, norms not counted."""
    return (mp.po.d * mp.po.bits + mp.pn.d * mp.pn.bits) / mp.d


def mixed_quantize(mp: MixedParams, X) -> dict:
    """Each part of every row quantized by its own quantizer."""
    X = np.asarray(X, dtype=np.float64)
    return {"o": quantize(mp.po, X[:, mp.out]), "n": quantize(mp.pn, X[:, mp.rest])}


def mixed_dequantize(mp: MixedParams, rows_o: dict, rows_n: dict) -> np.ndarray:
    """Both parts dequantized and written back to their channels."""
    xo = dequantize(mp.po, rows_o["idx"], rows_o["norm"], rows_o.get("z"), rows_o.get("rnorm"))
    xn = dequantize(mp.pn, rows_n["idx"], rows_n["norm"], rows_n.get("z"), rows_n.get("rnorm"))
    x = np.zeros((xo.shape[0], mp.d))
    x[:, mp.out] = xo
    x[:, mp.rest] = xn
    return x


def mixed_decode_attention(mk: MixedParams, mv: MixedParams, q, k_o: dict, k_n: dict, v_o: dict, v_n: dict,
                           seq_lens, Hkv: int, T_max: int, scale: float | None = None):
    """Plain softmax attention over the mixed-precision dequantized keys and values
    (rows ordered [B][Hkv][T_max]).  Returns (out [B, Hq, d], scores [B, Hq, T_max])."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    K = mixed_dequantize(mk, k_o, k_n).reshape(B, Hkv, T_max, d)
    V = mixed_dequantize(mv, v_o, v_n).reshape(B, Hkv, T_max, d)
    out = np.zeros((B, Hq, d))
    scores = np.full((B, Hq, T_max), np.nan)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            if L == 0:
                continue
            s = scale * (K[b, h // G, :L] @ q[b, h])
            scores[b, h, :L] = s
            w = np.exp(s - np.max(s))
            out[b, h] = (w / np.sum(w)) @ V[b, h // G, :L]
    return out, scores
