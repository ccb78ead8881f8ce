"""An independent float64 numpy statement of the DiT forward, for brute force on tiny inputs.

Written separately from the C++ oracle (einsum, explicit softmax over an explicit block mask,
a rotation written as a complex multiply) so that a mistake in one is unlikely to be repeated in the
other.  Used only on inputs of a handful of tokens.
"""
import numpy as np


def silu(v):
    return v / (1.0 + np.exp(-v))


def t_embed(t, t_dim):
    half = t_dim // 2
    k = np.arange(half, dtype=np.float64)
    f = np.exp(-np.log(10000.0) * k / half)
    return np.concatenate([np.cos(1000.0 * t * f), np.sin(1000.0 * t * f)])


def rope_angles(m, pos):
    """Angles [N, R/2]: per-axis blocks concatenated (t, h, w)."""
    cols = []
    for a in range(m["rope_axes"]):
        da = m["rope_dims"][a]
        inv = np.array([np.float32(m["rope_base"] ** (-2.0 * k / da)) for k in range(da // 2)], dtype=np.float64)
        cols.append(np.outer(pos[:, a], inv))
    return np.concatenate(cols, axis=1)


def rope(x, ang, H, Dh, R):
    """NeoX rotate_half as a complex multiply: z = (x_j + i x_{j+R/2}) * exp(i theta_j)."""
    x = x.reshape(x.shape[0], H, Dh).copy()
    half = R // 2
    z = (x[:, :, :half] + 1j * x[:, :, half:R]) * np.exp(1j * ang)[:, None, :]
    x[:, :, :half] = z.real
    x[:, :, half:R] = z.imag
    return x.reshape(x.shape[0], H * Dh)


def attention(q, k, v, cu, H, Dh):
    N = q.shape[0]
    mask = np.zeros((N, N), dtype=bool)
    for j in range(len(cu) - 1):
        mask[cu[j]:cu[j + 1], cu[j]:cu[j + 1]] = True
    qh = q.reshape(N, H, Dh)
    kh = k.reshape(N, H, Dh)
    vh = v.reshape(N, H, Dh)
    s = np.einsum("ihe,jhe->hij", qh, kh) / np.sqrt(Dh)
    s = np.where(mask[None], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("hij,jhe->ihe", p, vh).reshape(N, H * Dh)


def norm(x, m, g=None, b=None, kind=None):
    if (kind or m["norm"]) == "rms":
        y = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + m["norm_eps"])
        return y * (1.0 if g is None else g) + (0.0 if b is None else b)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    y = (x - mu) / np.sqrt(var + m["norm_eps"])
    return y * (1.0 if g is None else g) + (0.0 if b is None else b)


def forward(m, W, x_in, lay, t):
    d, F, H, Dh, R = m["hidden"], m["ffn_hidden"], m["n_heads"], m["head_dim"], m["rotary_dim"]
    cu, tags = lay["cu_seqlens"], lay["tags"].astype(np.int64)
    N = lay["n_tokens"]
    f64 = lambda a: None if a is None else np.asarray(a, dtype=np.float64)
    if m["io_channels"]:
        c = m["io_channels"]
        x = np.zeros((N, d))
        for j in range(len(cu) - 1):
            a, L = cu[j], cu[j + 1] - cu[j]
            xc = np.asarray(x_in[c * a:c * a + c * L], dtype=np.float64).reshape(c, L)
            x[a:a + L] = xc.T @ f64(W["glob"]["w_pre"]).T + f64(W["glob"]["b_pre"])
    else:
        x = np.asarray(x_in, dtype=np.float64).copy()
    ang = rope_angles(m, lay["pos"])
    nm = m["n_mod"]
    if m["adaln"]:
        # one timestep, or one per modality: the rows of modality i come from the embedding of t[i]
        ts = [t] * nm if np.ndim(t) == 0 else list(t)
        se = [silu(t_embed(ti, m["t_dim"])) for ti in ts]
    for l, bw in enumerate(W["blocks"]):
        B = {k: f64(v) for k, v in bw.items()}
        if m["adaln"]:
            wa = B["w_ada"].reshape(nm, 6 * d, -1)
            ba = B["b_ada"].reshape(nm, 6 * d)
            mod = np.stack([wa[i] @ se[i] + ba[i] for i in range(nm)]).reshape(nm, 6, d)[tags]  # [N, 6, d]
            y = norm(x, m) * (1 + mod[:, 1]) + mod[:, 0]
        else:
            y = norm(x, m, B.get("ln1_g"), B.get("ln1_b"))
        qkv = y @ B["w_qkv"].T + B["b_qkv"]
        if m.get("qkv_interleaved"):
            # per head [q_h | k_h | v_h]: view [N, H, 3 Dh] and split the last axis in three
            qh, kh, vh = np.split(qkv.reshape(N, H, 3 * Dh), 3, axis=2)
            q, k, v = qh.reshape(N, d), kh.reshape(N, d), vh.reshape(N, d)
        else:
            q, k, v = qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:]
        if m.get("qk_norm"):
            rmsn = lambda a: (a.reshape(N, H, Dh) / np.sqrt((a.reshape(N, H, Dh) ** 2).mean(axis=2, keepdims=True)
                                                          + m["norm_eps"])).reshape(N, d)
            q, k = rmsn(q), rmsn(k)
        q, k = rope(q, ang, H, Dh, R), rope(k, ang, H, Dh, R)
        o = attention(q, k, v, cu, H, Dh)
        upd = o @ B["w_o"].T + B["b_o"]
        x = x + (mod[:, 2] * upd if m["adaln"] else upd * (1.0 if B.get("res1") is None else B["res1"]))
        if m["adaln"]:
            y2 = norm(x, m) * (1 + mod[:, 4]) + mod[:, 3]
        else:
            y2 = norm(x, m, B.get("ln2_g"), B.get("ln2_b"))
        uv = y2 @ B["w_in"].T + B["b_in"]
        h = uv[:, :F] * silu(uv[:, F:])
        upd = h @ B["w_down"].T + B["b_down"]
        x = x + (mod[:, 5] * upd if m["adaln"] else upd * (1.0 if B.get("res2") is None else B["res2"]))
    if m["adaln"]:
        G = {k: f64(v) for k, v in W["glob"].items()}
        wf = G["w_ada_final"].reshape(nm, 2 * d, -1)
        bf = G["b_ada_final"].reshape(nm, 2 * d)
        mf = np.stack([wf[i] @ se[i] + bf[i] for i in range(nm)]).reshape(nm, 2, d)[tags]
        return norm(x, m) * (1 + mf[:, 1]) + mf[:, 0]
    G = {k: f64(v) for k, v in W["glob"].items()}
    y = norm(x, m, G.get("lnf_g"), G.get("lnf_b"), kind={"same": None, "rms": "rms", "ln": "ln"}[m.get("final_norm", "same")])
    if m["io_channels"]:
        c = m["io_channels"]
        out = np.zeros(c * N)
        for j in range(len(cu) - 1):
            a, L = cu[j], cu[j + 1] - cu[j]
            out[c * a:c * a + c * L] = (y[a:a + L] @ G["w_post"].T + G["b_post"]).T.reshape(-1)
        return out
    return y
