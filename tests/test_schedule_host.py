"""The projection schedule (host logic, no GPU): which schedule each matrix gets,
checked against the rule kd.h states, on the 8B shapes and around the rule's
edges.  The schedule depends on the shape and the SM count only, so every row's
arithmetic is the same for every batch size."""
import pytest

GROUP, STREAM = 1, 0
SMS = 152  # GB300


def expected_mode(groups, sms):
    if groups <= 2 * sms:
        return GROUP
    busiest = -(-groups // sms) * sms  # groups the busiest SM's share implies
    return GROUP if groups <= 8 * sms and busiest * 100 <= 105 * groups else STREAM


def share_brute_force(groups, kgroups, warps):
    """Most warps whose contiguous stage ranges meet in one row group."""
    stages = groups * kgroups
    owner = [0] * stages
    for w in range(warps):
        for t in range(w * stages // warps, (w + 1) * stages // warps):
            owner[t] = w
    return max(len(set(owner[g * kgroups:(g + 1) * kgroups])) for g in range(groups))


@pytest.mark.parametrize("rows,cols,mode", [
    (6144, 4096, GROUP),     # q|k|v: 192 groups, at most 2 per SM
    (4096, 4096, GROUP),     # o-proj: 128 groups
    (28672, 4096, GROUP),    # gate|up: 896 groups, 5.9 per SM (busiest 1.8% above the mean)
    (4096, 14336, GROUP),    # down
    (128256, 4096, STREAM),  # lm_head: 4008 groups, more than 8 per SM
])
def test_8b_shapes(kdlib, rows, cols, mode):
    got, warps, share = kdlib.kd_mmvq_schedule(rows, cols, SMS)
    assert got == mode
    if mode == STREAM:
        assert warps == min(8 * SMS, (rows // 32) * (cols // 128))
        assert share == share_brute_force(rows // 32, cols // 128, warps)
    else:
        assert share == 1


@pytest.mark.parametrize("groups", [1, 151, 152, 153, 304, 305, 456, 457, 608, 1216, 1217, 1520])
@pytest.mark.parametrize("kgroups", [1, 3, 32])
def test_rule_edges(kdlib, groups, kgroups):
    mode, warps, share = kdlib.kd_mmvq_schedule(groups * 32, kgroups * 128, SMS)
    assert mode == expected_mode(groups, SMS)
    assert warps == min(8 * SMS, groups * kgroups)
    if mode == STREAM:
        assert share == share_brute_force(groups, kgroups, warps)


@pytest.mark.parametrize("sms", [1, 8, 132, 148])
def test_other_sm_counts(kdlib, sms):
    for groups in (1, 2 * sms, 2 * sms + 1, 8 * sms + 1):
        assert kdlib.kd_mmvq_schedule(groups * 32, 256, sms)[0] == expected_mode(groups, sms)


def test_bad_shapes_are_refused(kdlib):
    for rows, cols, sms in ((16, 128, 152), (32, 64, 152), (33, 128, 152)):
        with pytest.raises(kdlib.KdError) as e:
            kdlib.kd_mmvq_schedule(rows, cols, sms)
        assert e.value.name == "KD_ERR_UNSUPPORTED"
    with pytest.raises(kdlib.KdError) as e:
        kdlib.kd_mmvq_schedule(32, 128, 0)
    assert e.value.name == "KD_ERR_INVALID_ARG"
