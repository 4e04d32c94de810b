"""Float64 CPU oracle for the sequence-tiled cross-entropy loss of the model's
last layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code
with the CUDA path, and the CUDA path never calls it.

What is computed, and where it is stated
----------------------------------------
* The pages' memory stack tiles the loss computation along the sequence, as
  it does the MLPs, so that no [sequence, vocabulary] buffer is created
  (memeeeeeex.com article, the stack section on Arctic sequence-length
  training; aipmzone.com article, the section from FSDP to Ulysses;
  liquidgold.cc talk transcript).  Each token's loss depends on that token's
  hidden state alone, so tiling changes memory, not the result: this oracle
  has no tiling.
* The loss itself is not spelled out on the pages.  Reading: the language-
  model cross entropy of the models they train, bias-free output projection
  W [V, hidden] (nn.Linear layout), natural log:
      z_i = h_i W^T,   lse_i = log sum_v exp(z_iv),   l_i = lse_i - z_i[t_i]
  and the reported loss is the mean of l_i over the S tokens.
* Backward of L = scale * sum_i l_i (scale = 1/S for the mean):
      dz_iv = scale * (softmax(z_i)_v - [v == t_i])
      dh = dz W,   dW = dz^T h
"""
import numpy as np


def logsumexp_rows(z):
    """log sum_v exp(z_v) of every row, shifted by the row max (no overflow)."""
    z = np.asarray(z, dtype=np.float64)
    m = z.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]


def loss_forward(h, W, targets):
    """Per-token loss l_i and log-sum-exp lse_i of logits z = h W^T."""
    h = np.asarray(h, dtype=np.float64)
    z = h @ np.asarray(W, dtype=np.float64).T
    lse = logsumexp_rows(z)
    t = np.asarray(targets, dtype=np.int64)
    return {"loss_rows": lse - z[np.arange(z.shape[0]), t], "lse": lse}


def loss_backward(h, W, targets, scale):
    """Gradients of L = scale * sum_i l_i with respect to h and W."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    z = h @ W.T
    lse = logsumexp_rows(z)
    p = np.exp(z - lse[:, None])
    p[np.arange(z.shape[0]), np.asarray(targets, dtype=np.int64)] -= 1.0
    dz = scale * p
    return {"dh": dz @ W, "dW": dz.T @ h}


def loss_total(h, W, targets, scale):
    """L = scale * sum_i l_i (the finite-difference pin's scalar)."""
    return float(scale * np.sum(loss_forward(h, W, targets)["loss_rows"]))
