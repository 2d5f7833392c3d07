"""Which prefill kernels a parity case runs through.

At head dimension 64 the library has two prefill kernels (two query tiles per work item, or
one) and picks one by the size of the call; a parity case at d = 64 runs through both, whatever
its size, by fixing the choice for the duration of the call.
"""
import contextlib


def d64_modes(d):
    """The kernel choices a case of head dimension d runs under."""
    return (1, 2) if d == 64 else (0,)


@contextlib.contextmanager
def d64_kernel(attn, mode):
    prev = attn.attn_fwd_set_d64_kernel(mode)
    try:
        yield
    finally:
        attn.attn_fwd_set_d64_kernel(prev)
