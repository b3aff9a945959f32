"""Algorithmic bytes and flops of one seam call (what the method must move).

Per token, each input read once and each output written once (the mHC seam
pages, "Realistic Bandwidth Ceiling": a post seam moves 1.678 GB at 16k rows of
H = 5120, i.e. 20 H bytes per token):

    R [4,H] bf16 read       8H      Y [H] bf16 read (post form)   2H
    R' [4,H] bf16 write     8H      norm [H] bf16 write           2H
    mxfp8: + H code bytes + H/32 scale bytes;  fp8 grid: + 2H (bf16 grid)

The identity (first-block) form reads R and writes the norm only: 10H.

Carried gates in (96 B/token) and gates out (96 B/token) and the per-call
weights (fn 4H x 24 fp32, gamma H bf16) are reported separately.
"""

GATE_BYTES_PER_TOKEN = 2 * (4 + 4 + 16) * 4


def stream_bytes_per_token(H: int, post: bool = True, out: str = "bf16", ident: bool = False) -> int:
    if ident and post:
        raise ValueError("the identity form has no post term")
    b = 8 * H + (0 if ident else 8 * H) + 2 * H + (2 * H if post else 0)
    if out == "mxfp8":
        b += H + H // 32
    elif out == "fp8_grid":
        b += 2 * H
    elif out != "bf16":
        raise ValueError(out)
    return b


def seam_bytes(T: int, H: int, post: bool = True, out: str = "bf16", gates: bool = False,
               ident: bool = False) -> int:
    b = T * stream_bytes_per_token(H, post, out, ident)
    if gates:
        b += T * GATE_BYTES_PER_TOKEN
    return b


def seam_flops_per_token(H: int, post: bool = True) -> int:
    """Post-mix 40H (32H without Y), sum of squares 8H, projection 192H,
    collapse 8H, x sum of squares and norm 4H."""
    return (40 if post else 32) * H + 8 * H + 192 * H + 8 * H + 4 * H
