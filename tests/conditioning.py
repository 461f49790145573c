"""The conditioning reading used where an input is ill-conditioned for bf16
Newton-Schulz (test helper; imports the oracle).

The pages fix no order for the fp32 sums of the products, so the oracle's
ascending order and the descending order are equally valid.  An input is
well-conditioned when the oracle's O under the two orders agree within half
the contract (relative Frobenius 5e-3, per-element 1e-2): there any other
summation order, the tensor cores' included, is held to the contract itself.
Where the two legal orders alone differ by more, no implementation that sums
in another order can promise the contract, and the bound becomes the contract
plus the oracle's own spread between the two orders.
"""
import oracle
from tests.gpu_util import ABS_TOL, REL_TOL, compare_o


def order_spread(step_fn):
    """(relative, absolute) distance between the O that ``step_fn()`` returns
    under the oracle's two summation orders."""
    o_asc = step_fn()
    with oracle.descending_sums():
        o_desc = step_fn()
    return compare_o(o_desc, o_asc)


def bound_for(spread):
    """(rel bound, abs bound, well_conditioned) for an input with this spread."""
    rel_s, abs_s = spread
    if rel_s <= REL_TOL / 2 and abs_s <= ABS_TOL / 2:
        return REL_TOL, ABS_TOL, True
    return REL_TOL + rel_s, ABS_TOL + abs_s, False
