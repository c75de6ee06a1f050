"""Seeded synthetic inputs for the Gated Subspace Inference (GSI) linear map.

This module is shared by the tests, the oracle side and the CUDA side, and
therefore holds none of the method's arithmetic: it never forms g, r, rho, a
gate or an output, and never forms the cached image M.  It only draws

* weights       W ~ N(0, 1/d), stored bf16;
* bases         V_k = the first k columns of Q from QR of a seeded Gaussian
                d x (k+m) matrix (signs fixed so diag(R) > 0), stored bf16;
                the remaining m columns of Q are kept in fp64 as residual
                directions orthogonal to span(V_k);
* activations   x = a + s b, with a a random vector in a fixed 200-dimensional
                subspace of span(V_k) and b a random combination of the m
                residual directions, s chosen so that the fp64 construction
                has residual ratio rho* exactly; rho* is drawn per token
                uniformly in [0.9, 1.1] x a nominal value.  Stored bf16.

Which tokens are slow (large rho*) is drawn as exact counts at seeded
positions.  Workload shapes follow the page "Technical summary: Gated
Subspace Inference for transformer acceleration", section 4 (GPT-2 124M,
GPT-J 6B and OPT 6.7B at k = 256, eps = 0.10, batch size 1); the trained
weights and text those experiments used are not available, and these
synthetic draws of the same shapes stand in for them.

All bf16 values are numpy ``uint16`` bit patterns (or torch bf16 tensors for
large weights drawn on a device).  bf16 rounding here is this module's own
round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

# --------------------------------------------------------------------------
# bf16 bit patterns
# --------------------------------------------------------------------------


def to_bf16_bits(a) -> np.ndarray:
    """fp64 (or fp32) array -> bf16 bit patterns, round to nearest even.

    Finite values only (the generator never makes others).  One rounding
    from the fp64 value: with v = m 2^e (0.5 <= |m| < 1), the bf16 quantum is
    2^(e-8) (never below 2^-133); rint() rounds ties to even.
    """
    v = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(v)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(v, -q)), q)
    f = r.astype(np.float32)  # exact: r has <= 8 significant bits
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(t) for t in tags]))


# --------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------


def gaussian_weights(d_out: int, d: int, seed: int, tag: int = 0,
                     device: Optional[str] = None):
    """W ~ N(0, 1/d), shape d_out x d, stored bf16.

    device=None: numpy draw, returns uint16 bit patterns.
    device="cuda"/"cpu": torch draw on that device with a seeded torch
    generator, returns a torch.bfloat16 tensor (used for multi-GB stacks).
    The two routes draw different numbers for the same seed; each route is
    reproducible on its own.
    """
    scale = 1.0 / math.sqrt(d)
    if device is None:
        rng = _rng(seed, 0xA1, tag)
        out = np.empty((d_out, d), dtype=np.uint16)
        rows = max(1, (1 << 22) // max(d, 1))
        for r0 in range(0, d_out, rows):
            r1 = min(d_out, r0 + rows)
            z = rng.standard_normal((r1 - r0, d), dtype=np.float32)
            z *= np.float32(scale)
            u = z.view(np.uint32)
            out[r0:r1] = ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
        return out
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + 0xA1 * 7919 + int(tag)) & 0x7FFFFFFFFFFFFFFF)
    w = torch.empty((d_out, d), dtype=torch.bfloat16, device=device)
    rows = max(1, (1 << 26) // max(d, 1))
    for r0 in range(0, d_out, rows):
        r1 = min(d_out, r0 + rows)
        z = torch.randn((r1 - r0, d), generator=g, device=device, dtype=torch.float32)
        w[r0:r1] = (z * scale).to(torch.bfloat16)
    return w


# --------------------------------------------------------------------------
# Bases
# --------------------------------------------------------------------------


@dataclass
class Basis:
    """An orthonormal rank-k basis and m residual directions, fp64 and bf16."""
    Q: np.ndarray          # d x k, fp64, orthonormal columns (before rounding)
    perp: np.ndarray       # d x m, fp64, orthonormal, orthogonal to Q
    V_bits: np.ndarray     # d x k, bf16 bit patterns of Q (the stored V_k)
    sub: np.ndarray        # k x n_sub, fp64 orthonormal: the activation subspace inside span(V_k)

    @property
    def d(self) -> int:
        return self.Q.shape[0]

    @property
    def k(self) -> int:
        return self.Q.shape[1]


def _qr_signed(A: np.ndarray) -> np.ndarray:
    Q, R = np.linalg.qr(A)
    s = np.sign(np.diag(R))
    s[s == 0] = 1.0
    return Q * s


def _n_perp(d: int, k: int) -> int:
    return int(min(64, d - k))


def random_basis(d: int, k: int, seed: int, tag: int = 0, n_sub: int = 200) -> Basis:
    """V_k = Q of QR(seeded Gaussian), stored bf16; plus residual directions."""
    rng = _rng(seed, 0xB2, tag)
    m = _n_perp(d, k)
    Q = _qr_signed(rng.standard_normal((d, k + m)))
    return _finish_basis(Q[:, :k], Q[:, k:], rng, n_sub)


def coherent_next_basis(prev: Basis, seed: int, tag: int, mix: float = 0.3,
                        n_sub: int = 200) -> Basis:
    """Next layer's basis: QR(V_prev + mix * E), E ~ N(0, 1/d) entrywise.

    The perturbation is read relative to unit basis columns (entries of
    N(0, 1/d) have column norm ~1), which keeps adjacent subspaces close, as
    the page's depth-coherence observation describes (section 2.3).
    """
    rng = _rng(seed, 0xC3, tag)
    d, k = prev.Q.shape
    m = _n_perp(d, k)
    E = rng.standard_normal((d, k)) / math.sqrt(d)
    Q = _qr_signed(np.concatenate([prev.Q + mix * E, rng.standard_normal((d, m))], axis=1))
    return _finish_basis(Q[:, :k], Q[:, k:], rng, n_sub)


def _finish_basis(Qk: np.ndarray, perp: np.ndarray, rng, n_sub: int) -> Basis:
    k = Qk.shape[1]
    n_sub = min(n_sub, k)
    sub = _qr_signed(rng.standard_normal((k, n_sub)))
    return Basis(Q=np.ascontiguousarray(Qk), perp=np.ascontiguousarray(perp),
                 V_bits=to_bf16_bits(Qk), sub=sub)


# --------------------------------------------------------------------------
# Activations
# --------------------------------------------------------------------------


def tokens(basis: Basis, rho_star: np.ndarray, seed: int, tag: int = 0,
           scale: float = 1.0) -> np.ndarray:
    """T activations (bf16 bits, T x d) with fp64 residual ratio rho_star[t].

    x = a + s b: a = Q (sub c), c ~ N(0, I); b = perp z, z ~ N(0, I);
    s = rho* ||a|| / (sqrt(1 - rho*^2) ||b||), so ||s b|| / ||x|| = rho* in
    fp64 because a is orthogonal to b.  rho* = 1 gives a pure residual token.
    Each token is then scaled to norm ~ scale * sqrt(d) times a log-normal
    factor, and rounded to bf16 (which moves rho by ~1e-3 at most).
    """
    rho_star = np.asarray(rho_star, dtype=np.float64)
    T = rho_star.shape[0]
    d, k = basis.Q.shape
    rng = _rng(seed, 0xD4, tag)
    c = rng.standard_normal((T, basis.sub.shape[1]))
    a = (c @ basis.sub.T) @ basis.Q.T                 # T x d, in span(V_k)
    m = basis.perp.shape[1]
    if m > 0:
        z = rng.standard_normal((T, m))
        b = z @ basis.perp.T                          # T x d, orthogonal to V_k
    else:
        b = np.zeros((T, d))
    na = np.linalg.norm(a, axis=1)
    nb = np.linalg.norm(b, axis=1)
    x = np.empty((T, d))
    for t in range(T):
        p = rho_star[t]
        if p >= 1.0:
            x[t] = b[t] / nb[t]
        elif p <= 0.0 or nb[t] == 0.0:
            x[t] = a[t] / na[t]
        else:
            s = p * na[t] / (math.sqrt(1.0 - p * p) * nb[t])
            x[t] = a[t] + s * b[t]
            x[t] /= np.linalg.norm(x[t])
    amp = scale * math.sqrt(d) * np.exp(0.25 * rng.standard_normal(T))
    return to_bf16_bits(x * amp[:, None])


def rho_targets(n: int, nominal_fast: float, nominal_slow: float,
                slow_mask: np.ndarray, seed: int, tag: int = 0) -> np.ndarray:
    """Per-token rho*: nominal x U[0.9, 1.1], slow or fast nominal by mask."""
    rng = _rng(seed, 0xE5, tag)
    u = rng.uniform(0.9, 1.1, size=n)
    return np.where(slow_mask, nominal_slow, nominal_fast) * u


def slow_positions(n: int, n_slow: int, seed: int, tag: int = 0) -> np.ndarray:
    """Boolean mask with exactly n_slow True entries at seeded positions."""
    rng = _rng(seed, 0xF6, tag)
    mask = np.zeros(n, dtype=bool)
    if n_slow > 0:
        mask[rng.choice(n, size=n_slow, replace=False)] = True
    return mask


# --------------------------------------------------------------------------
# Workload configurations (shapes from the page's section 4 models)
# --------------------------------------------------------------------------

CONFIG_SEED_BASE = 20260000


@dataclass
class LinearSpec:
    """One gated linear: its shapes, threshold and token mix."""
    name: str
    d_out: int
    d: int
    k: int
    eps: float
    rho_fast: float
    rho_slow: float


@dataclass
class Workload:
    name: str
    seed: int
    linears: List[LinearSpec]
    T: int                       # tokens per forward call
    extra: Dict = field(default_factory=dict)


def gpt2_qkv(T: int = 64, n_slow: int = 6) -> Workload:
    """GPT-2-small-shaped QKV linear (768 -> 2304), k = 256, eps = 0.10,
    T = 64 with 10% slow tokens (round(6.4) = 6); fast rho* ~ 0.03, slow ~ 0.3."""
    return Workload("gpt2_qkv_T64", CONFIG_SEED_BASE + 0,
                    [LinearSpec("qkv", 2304, 768, 256, 0.10, 0.03, 0.3)], T,
                    dict(n_slow=n_slow))


def gptj_layer(n_tokens: int = 512) -> Workload:
    """GPT-J-6B-shaped decoder layer at T = 1 decode.

    q, k, v and fc_in read the same input, so they form one stacked linear
    (4096 -> 3*4096 + 16384 = 28672) with one V_k and one gate per token; the
    output projection (4096 -> 4096) and fc_out (16384 -> 4096) have their
    own bases.  k = 256, eps = 0.10; 512 sequential tokens, exactly one of
    them slow (round(0.002 * 512) = 1) in all three linears; fast rho* ~ 0.05,
    slow rho* ~ 0.4.
    """
    lin = [LinearSpec("qkv_fc_in", 28672, 4096, 256, 0.10, 0.05, 0.4),
           LinearSpec("out_proj", 4096, 4096, 256, 0.10, 0.05, 0.4),
           LinearSpec("fc_out", 4096, 16384, 256, 0.10, 0.05, 0.4)]
    return Workload("gptj_layer_decode", CONFIG_SEED_BASE + 1, lin, 1,
                    dict(n_tokens=n_tokens, n_slow=max(1, round(0.002 * n_tokens))))


def gptj_stack(n_layers: int = 28, n_steps: int = 256) -> Workload:
    """28 GPT-J layers of the decode layer's three linears, depth-coherent
    bases, 256 decode steps; slow draws per (step, layer, linear) as an exact
    count round(0.002 * steps * layers * 3) at seeded positions."""
    w = gptj_layer()
    total = n_steps * n_layers * 3
    return Workload("gptj_stack_decode", CONFIG_SEED_BASE + 2, w.linears, 1,
                    dict(n_layers=n_layers, n_steps=n_steps,
                         n_slow=round(0.002 * total)))


def opt_mlp(n_layers: int = 32, n_steps: int = 256,
            slow_fraction: float = 0.0) -> Workload:
    """OPT-6.7B-shaped MLP linears fc1 (4096 -> 16384) and fc2 (16384 -> 4096),
    32 layers, k = 256, eps = 0.05, T = 1; slow fraction f as an exact count
    over (step, layer, linear); fast rho* ~ 0.02, slow rho* ~ 0.3."""
    lin = [LinearSpec("fc1", 16384, 4096, 256, 0.05, 0.02, 0.3),
           LinearSpec("fc2", 4096, 16384, 256, 0.05, 0.02, 0.3)]
    total = n_steps * n_layers * 2
    return Workload(f"opt_mlp_f{int(round(slow_fraction * 100))}",
                    CONFIG_SEED_BASE + 3, lin, 1,
                    dict(n_layers=n_layers, n_steps=n_steps,
                         slow_fraction=slow_fraction,
                         n_slow=int(round(slow_fraction * total))))


def batched_prefill(T: int = 512) -> Workload:
    """Batched gated linear: T = 512 tokens, W 16384 x 4096, k = 256,
    eps = 0.10; 30% slow (round(0.3 * 512) = 154, rho* ~ 0.3) at random
    positions, 70% fast (rho* ~ 0.04)."""
    return Workload("batched_T512", CONFIG_SEED_BASE + 4,
                    [LinearSpec("proj", 16384, 4096, 256, 0.10, 0.04, 0.3)], T,
                    dict(n_slow=int(round(0.3 * T))))


@dataclass
class LinearInputs:
    """Inputs of one gated linear: W (bf16), basis, tokens (bf16), slow mask."""
    spec: LinearSpec
    W: object                 # uint16 ndarray or torch.bfloat16 tensor
    basis: Basis
    X_bits: np.ndarray        # T x d bf16 bits
    slow_mask: np.ndarray     # T bools (the intended branch; rho* decides)

    @property
    def V_bits(self) -> np.ndarray:
        return self.basis.V_bits


def make_linear_inputs(spec: LinearSpec, T: int, n_slow: int, seed: int,
                       tag: int = 0, w_device: Optional[str] = None,
                       basis: Optional[Basis] = None,
                       slow_mask: Optional[np.ndarray] = None) -> LinearInputs:
    """Draw W, V_k and T tokens for one linear (exact slow count)."""
    W = gaussian_weights(spec.d_out, spec.d, seed, tag, device=w_device)
    if basis is None:
        basis = random_basis(spec.d, spec.k, seed, tag)
    if slow_mask is None:
        slow_mask = slow_positions(T, n_slow, seed, tag)
    rs = rho_targets(T, spec.rho_fast, spec.rho_slow, slow_mask, seed, tag)
    X = tokens(basis, rs, seed, tag)
    return LinearInputs(spec, W, basis, X, slow_mask)


# --------------------------------------------------------------------------
# Calibration activations
# --------------------------------------------------------------------------


@dataclass
class CalibrationSet:
    """n calibration tokens with a planted spectrum.

    X_bits  n x d bf16 bits, the tokens;
    U       d x r fp64 orthonormal, the planted directions (descending scale);
    sigma   r planted scales; token t is U (sigma * c_t) + noise, c_t ~ N(0, I),
            then rescaled, so the population second moment has eigenvectors
            U with eigenvalues proportional to sigma^2 above an isotropic floor.
    """
    X_bits: np.ndarray
    U: np.ndarray
    sigma: np.ndarray


def planted_scales(r: int, k: int, decay: float = 0.5, gap: float = 0.5) -> np.ndarray:
    """sigma_j = (1 + j)^-decay for j < k and gap * (1 + j)^-decay for j >= k:
    a power-law spectrum with a step of gap^2 between the k-th and (k+1)-th
    eigenvalue of the second moment."""
    j = np.arange(r, dtype=np.float64)
    s = (1.0 + j) ** (-decay)
    s[k:] *= gap
    return s


def calibration_activations(n: int, d: int, k: int, seed: int, tag: int = 0,
                            r: Optional[int] = None, decay: float = 0.5,
                            gap: float = 0.5, noise: float = 0.02,
                            U: Optional[np.ndarray] = None) -> CalibrationSet:
    """Seeded stand-in for the activations of one calibration sequence.

    x_t = a_t (U (sigma * c_t) + noise * z_t), with c_t ~ N(0, I_r),
    z_t ~ N(0, I_d / d) (unit expected norm), U d x r orthonormal (QR of a
    seeded Gaussian, or the given U), sigma from planted_scales(r, k, decay,
    gap), and a_t = sqrt(d / sum(sigma^2)) * exp(0.25 N(0, 1)) so that entries
    are O(1) with a log-normal spread of token norms.  r defaults to
    min(d, 2k).
    """
    if r is None:
        r = min(d, 2 * k) if U is None else U.shape[1]
    rng = _rng(seed, 0xCA, tag)
    if U is None:
        U = _qr_signed(rng.standard_normal((d, r)))
    sigma = planted_scales(r, k, decay, gap)
    c = rng.standard_normal((n, r)) * sigma
    x = c @ U.T
    if noise > 0:
        x += (noise / math.sqrt(d)) * rng.standard_normal((n, d))
    amp = math.sqrt(d / float(np.sum(sigma ** 2))) * np.exp(0.25 * rng.standard_normal(n))
    return CalibrationSet(X_bits=to_bf16_bits(x * amp[:, None]), U=U, sigma=sigma)


def calibration_start(d: int, k: int, seed: int, tag: int = 0) -> np.ndarray:
    """The random start block of the basis iteration: d x k entries
    ~ N(0, 1/d), bf16 bits (the layout of V_k)."""
    rng = _rng(seed, 0xCB, tag)
    return to_bf16_bits(rng.standard_normal((d, k)) / math.sqrt(d))


def calibration_gptj(n: int = 2048) -> Dict:
    """Calibration of one GPT-J-6B-shaped linear input (d = 4096, k = 256)
    from one 2048-token sequence (GPT-J's context length); 8 iterations."""
    return dict(name="calibrate_gptj_d4096", seed=CONFIG_SEED_BASE + 5, n=n, d=4096,
                k=256, iters=8)


def calibration_cascade(n_layers: int, n: int, d: int, k: int, seed: int, mix: float = 0.3,
                        **kw) -> List[CalibrationSet]:
    """Calibration tokens of n_layers consecutive layers whose planted
    directions are depth-coherent: U_{l+1} = QR(U_l + mix * E_l), E_l ~
    N(0, 1/d) per entry (relative to unit columns, as coherent_next_basis),
    each layer's tokens drawn by calibration_activations with its own U and
    seed tag.  With mix = 0.3 adjacent layers' planted subspaces have mean
    principal-angle cosines near 0.96, in line with the page's observation of
    > 0.90 in deeper layers (section 2.3)."""
    r = kw.pop("r", None) or min(d, 2 * k)
    rng = _rng(seed, 0xCC)
    U = _qr_signed(rng.standard_normal((d, r)))
    out = []
    for layer in range(n_layers):
        out.append(calibration_activations(n, d, k, seed, tag=layer, U=U, **kw))
        E = rng.standard_normal((d, r)) / math.sqrt(d)
        U = _qr_signed(U + mix * E)
    return out


def sweep_activations(T: int, d: int, seed: int, r: int = 1024, decay: float = 1.0,
                      noise: float = 0.02, tag: int = 0) -> CalibrationSet:
    """Tokens for operating-point sweeps: a gapless power-law spectrum
    sigma_j = (1 + j)^-decay over r planted directions (decay 1 puts about
    0.6 / k of a token's energy outside the top k directions, so rho ~ 0.05 at
    k = 256: the concentration the page reports for GPT-J, 99.8% of tokens
    below eps = 0.10), plus the isotropic noise floor of
    calibration_activations.  U[:, :k] is the population top-k basis."""
    return calibration_activations(T, d, r, seed, tag=tag, r=r, decay=decay, gap=1.0,
                                   noise=noise)
