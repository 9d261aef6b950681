"""Per-configuration counts of the parity exclusions.

Where floating point may legitimately decide a discrete outcome differently on the two
sides, the parity tests exclude that unit and count it:
  near_tie    a draft position whose oracle top-2 biased-logit gap is within the logit
              tolerance (4 * (atol + rtol * |top|)); `flip` counts those where the GPU
              actually chose the other token (the oracle then continues from the GPU's
              token, teacher-forced)
  accept      an accept test with |u - p/q| inside the decision window (1e-5, widened by
              the propagated logit difference when the two sides' draft logits differ)
  draw        a Gumbel-max draw whose gap to the runner-up is within the oracle's binary32
              error bound
  confidence  a confidence decision within 1e-4 of the threshold
The conftest prints the table at the end of the session.
"""
RECORDS = []


def record(config, unit, compared, **counts):
    RECORDS.append((config, unit, int(compared), {k: int(v) for k, v in counts.items()}))


def summary_lines():
    if not RECORDS:
        return []
    keys = []
    for _, _, _, c in RECORDS:
        for kk in c:
            if kk not in keys:
                keys.append(kk)
    lines = ["parity exclusions per configuration (counted, then excluded):",
             "  %-44s %-10s %8s " % ("configuration", "unit", "compared") + " ".join("%10s" % kk for kk in keys)]
    for cfg, unit, n, c in RECORDS:
        lines.append("  %-44s %-10s %8d " % (cfg[:44], unit, n) + " ".join("%10d" % c.get(kk, 0) for kk in keys))
    return lines
