"""Float64 CPU oracle for the sequence-tiled MLP of the decoder layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path, and the CUDA path never calls it.

What is computed, and where it is stated
----------------------------------------
* The pages' memory stack tiles the element-wise parts of the layer (the
  MLPs and the loss) along the sequence, so that no buffer as long as the
  sequence is ever created (memeeeeeex.com article, the stack section on
  Arctic sequence-length training; aipmzone.com article, the section from
  FSDP to Ulysses; talk transcript on liquidgold.cc; dimanyen.com summary,
  "Core stack", layer 5).  Tiling rows changes memory, not the result: each
  token's MLP output depends on that token alone.  So this oracle has no
  tiling; it computes the MLP by its definition over all rows at once, and
  tile invariance is a property the tests check.
* The MLP itself is not spelled out on the pages.  Reading: the standard
  bias-free SwiGLU MLP of the Llama / Qwen3 models the pages train
  ("Results": Llama3-8B, Qwen3-32B), with nn.Linear weight layouts
      g = x Wg^T,  u = x Wu^T          (Wg, Wu: [ffn, hidden])
      a = silu(g) * u,  silu(v) = v * sigmoid(v)
      y = a Wd^T                       (Wd: [hidden, ffn])
* Backward of L = sum(y * dy), by the chain rule written out:
      da = dy Wd,  dWd = dy^T a
      dg = da * u * silu'(g),  silu'(v) = s (1 + v (1 - s)),  s = sigmoid(v)
      du = da * silu(g)
      dx = dg Wg + du Wu,  dWg = dg^T x,  dWu = du^T x

Everything is float64; inputs are converted exactly from their bf16 storage
by the caller.
"""
import numpy as np


def sigmoid(v):
    """Logistic function 1 / (1 + e^-v), evaluated without overflow for large
    |v| (the exponential is only ever taken of a non-positive number)."""
    v = np.asarray(v, dtype=np.float64)
    e = np.exp(-np.abs(v))
    return np.where(v >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def silu(v):
    """SiLU (swish): v * sigmoid(v)."""
    v = np.asarray(v, dtype=np.float64)
    return v * sigmoid(v)


def silu_grad(v):
    """d silu / dv = s + v s (1 - s) with s = sigmoid(v)."""
    v = np.asarray(v, dtype=np.float64)
    s = sigmoid(v)
    return s * (1.0 + v * (1.0 - s))


def mlp_forward(x, Wg, Wu, Wd):
    """SwiGLU MLP of every row of x [S, hidden]: returns the intermediates
    g, u, a ([S, ffn]) and the output y [S, hidden]."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ np.asarray(Wg, dtype=np.float64).T
    u = x @ np.asarray(Wu, dtype=np.float64).T
    a = silu(g) * u
    y = a @ np.asarray(Wd, dtype=np.float64).T
    return {"g": g, "u": u, "a": a, "y": y}


def mlp_backward(x, Wg, Wu, Wd, dy):
    """Gradients of L = sum(y * dy) with respect to x and the three weights
    (the chain rule above), plus the intermediates the GPU path stores."""
    x = np.asarray(x, dtype=np.float64)
    Wg = np.asarray(Wg, dtype=np.float64)
    Wu = np.asarray(Wu, dtype=np.float64)
    Wd = np.asarray(Wd, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    f = mlp_forward(x, Wg, Wu, Wd)
    g, u, a = f["g"], f["u"], f["a"]
    da = dy @ Wd
    dg = da * u * silu_grad(g)
    du = da * silu(g)
    return {"dx": dg @ Wg + du @ Wu, "dWg": dg.T @ x, "dWu": du.T @ x, "dWd": dy.T @ a,
            "dg": dg, "du": du, "a": a, "y": f["y"]}


def mlp_loss(x, Wg, Wu, Wd, dy):
    """L = sum(y * dy): the scalar whose gradient mlp_backward returns (used
    by the finite-difference pin)."""
    return float(np.sum(mlp_forward(x, Wg, Wu, Wd)["y"] * np.asarray(dy, dtype=np.float64)))
